/* moe_fp8.h -- C ABI of the GB300 (sm_103a) routed FP8 block-scaled MoE FFN library.
 *
 * One layer of a routed mixture-of-experts FFN whose expert weights are FP8 E4M3 with one
 * FP32 scale per 128x128 block:
 *   route      softmax + top-k over BF16 router logits           (moe_route)
 *   prepare    hidden -> FP8 per token per 128 columns; counting-sort permutation of the
 *              (token, slot) pairs into expert-contiguous tiles     (moe_fp8_prepare)
 *   gate/up    block-scaled grouped GEMM + fused SiLU(gate)*up with requantisation to FP8
 *              at one scale per routed row per 128 columns          (moe_fp8_gate_up)
 *   down       block-scaled grouped GEMM                            (moe_fp8_down)
 *   combine    top-k weighted sum in slot order, no atomics         (moe_fp8_combine)
 * moe_fp8_forward runs prepare -> gate/up -> down -> combine, or, for at most 64 routed
 * rows (M * top_k), gate/up (quantising hidden itself) -> down fused with the combine.
 * Between 65 and 256 routed rows gate/up and down run over groups of up to 16 sorted rows
 * of one expert (each expert's weights read once per group); above, over 128-row tiles.
 * moe_fp8_route_forward_one_launch runs routing and the whole layer as a single kernel.
 *
 * Sources (web pages; each entry point names the passage that defines it):
 *   [NK]   "NetraRuntime/netra-kernel" README
 *   [NKL]  "NetraRuntime/netra-kernel" older kernel-lab README
 *   [ARCH] netra-kernel docs/compiler/architecture.md
 *   [AMDK] "Inferact/amd-kernels" README
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller, 16-byte aligned, with
 *     the row-major layouts stated below (moe_fp8_route_forward_host takes its hidden and
 *     out in host memory; moe_fp8_read_status writes a host word). The library never
 *     allocates, frees or synchronises; host<->device copies happen only in those two calls,
 *     enqueued on the caller's stream ([NKL] "Design": the dispatch path avoids allocation,
 *     synchronisation, filesystem access, environment parsing and symbol lookup).
 *   - Work is enqueued on `stream` (0 = legacy default stream) and returns at once.
 *     Nothing in the library keeps per-call state between calls: two calls on different
 *     streams with different workspaces may run concurrently ([ARCH], caller-local
 *     kernel arguments). Calls sharing one workspace must be ordered on one stream.
 *   - Host-side validation runs before any launch and returns MOE_ERR_INVALID_ARG (null or
 *     misaligned pointer, M out of range), MOE_ERR_UNSUPPORTED (shape outside the compiled
 *     set: [NK] exact contracts, no approximate dispatch; there is no fallback path) or
 *     MOE_ERR_WORKSPACE (workspace too small). A launch error is MOE_ERR_LAUNCH.
 *   - Errors the device finds (an expert id outside [0, E), a bounded wait that ran out)
 *     never trap: they set bits of a status word in the workspace, read back with
 *     moe_fp8_read_status.
 *   - Numerics (the contract; [NK] lists accumulation, rounding and reduction order as
 *     part of an operation's identity): see each call.
 */
#ifndef MOE_FP8_H_
#define MOE_FP8_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_WORKSPACE = 3,
  MOE_ERR_LAUNCH = 4
} moe_status_t;

/* Device status bits (moe_fp8_read_status). */
#define MOE_STATUS_BAD_EXPERT_ID 0x1u /* an id < 0 or >= E was skipped (contributes 0) */
#define MOE_STATUS_WAIT_TIMEOUT 0x2u  /* a bounded device wait gave up; outputs invalid */

/* Layer shape. hidden (H) is a multiple of 256 (the down GEMM's 256-wide output blocks) with
 * 256 <= H <= 8192; inter (I) is a multiple of 128 (the block-scale grid) with
 * 128 <= I <= 4096; num_experts (E) in {8,16,32,64,128,256}; 1 <= top_k (K) <= min(E,16).
 * max_tokens (1 <= max_tokens <= 2^20 / K) bounds M for every call that uses one workspace.
 * Any other shape is MOE_ERR_UNSUPPORTED (moe_fp8_workspace_bytes returns 0). */
typedef struct {
  int32_t hidden;
  int32_t inter;
  int32_t num_experts;
  int32_t top_k;
  int32_t max_tokens;
} moe_fp8_shape_t;

/* Library version string (static storage). */
const char* moe_fp8_version(void);

/* Bytes of caller-owned device workspace that moe_fp8_forward and the stage calls need
 * for this shape (pure host arithmetic; 0 if the shape is unsupported). [ARCH]: the
 * standalone graph owns its deterministic static intermediates. */
size_t moe_fp8_workspace_bytes(const moe_fp8_shape_t* shape);

/* Clear the workspace's status word and the arrival counters of
 * moe_fp8_route_forward_one_launch. Call once after allocating a workspace (enqueued on
 * `stream`); every call leaves the counters at zero, and every other region is fully
 * rewritten by each forward call. */
moe_status_t moe_fp8_workspace_init(void* workspace, size_t workspace_bytes,
                                    const moe_fp8_shape_t* shape, cudaStream_t stream);

/* Router: [NK] capability table (BF16 routing) and prefill-pair section ("semantic
 * routing" stage of the routed MoE producer).
 *   hidden    BF16 [M][H] row-major
 *   router_w  BF16 [H][E] (E contiguous)
 *   bias      FP32 [E] added to every logit, or NULL
 *   topk_ids  int32 [M][K] out; slot j holds the expert with the j-th largest logit
 *             (ties to the lower expert index)
 *   topk_w    FP32 [M][K] out; renormalize != 0: softmax over the K selected logits,
 *             else the softmax over all E logits read at the selected experts
 * logit[t][e] = sum over 128-wide chunks c ascending of an FP32 fma chain over the
 * chunk's k ascending (from 0), then + bias[e]. Top-k ids are a pure function of these
 * logits. M = 0 is a no-op. Needs no workspace.
 * router_w and bias are layer parameters: they are read while the kernel launched just
 * before this call on `stream` may still be running (programmatic dependent launch), so
 * that kernel must not write them. hidden is read only after it has completed. */
moe_status_t moe_route(const void* hidden, const void* router_w, const float* bias, int32_t M,
                       const moe_fp8_shape_t* shape, int32_t renormalize, int32_t* topk_ids,
                       float* topk_w, cudaStream_t stream);

/* RMSNorm in front of the layer ([NKL] "Repository layout": gfx950 normalisation and
 * quantisation fusions; the Qwen3.6 RMSNorm patch listed beside it). The pages fix neither the
 * epsilon nor the weight convention; this library computes, per token row,
 *   y[k] = bf16_rn((x[k] * r) * norm_weight[k]),   r = 1 / sqrt(ss / H + eps),
 * where ss = sum of x[k]^2 in the router's order (an FP32 fma chain over each 128-wide chunk,
 * k ascending from 0, the chunk partials added in ascending order) and every other step is one
 * correctly rounded FP32 operation (division by H, + eps, square root, 1 / s, two multiplies).
 *   hidden       BF16 [M][H] (the un-normalised rows)
 *   norm_weight  BF16 [H], 16-byte aligned
 *   eps          finite and > 0 (else MOE_ERR_INVALID_ARG)
 * The norm entry points below apply this transform inside their own kernels (the router and
 * the hidden quantisers form r themselves; nothing is written between them) and are otherwise
 * the calls without "norm": moe_norm_route == moe_route(y), moe_fp8_norm_forward ==
 * moe_fp8_forward(y), moe_fp8_norm_route_forward == moe_fp8_route_forward(y), bit for bit.
 * moe_rmsnorm writes y itself (BF16 [M][H], out may not alias hidden) for callers that also
 * need it. M = 0 is a no-op; M <= shape->max_tokens. */
moe_status_t moe_rmsnorm(const void* hidden, const void* norm_weight, float eps, int32_t M, void* out,
                         const moe_fp8_shape_t* shape, cudaStream_t stream);
moe_status_t moe_norm_route(const void* hidden, const void* norm_weight, float eps, const void* router_w,
                            const float* bias, int32_t M, const moe_fp8_shape_t* shape, int32_t renormalize,
                            int32_t* topk_ids, float* topk_w, cudaStream_t stream);

/* The routed expert FFN ([ARCH] accepted M=1 MoE objects: gate/up, SiLU+quant and
 * down/reduce; [NK] prefill-pair section: producer stages plus a separate route reducer
 * with its own fixed reduction order; [AMDK] reduction rule: fixed order, no atomics).
 *   hidden     BF16 [M][H]
 *   topk_ids   int32 [M][K]     (ids outside [0,E) are skipped and flagged)
 *   topk_w     FP32 [M][K]
 *   w13        E4M3 [E][2I][H]  rows 0..I-1 gate, I..2I-1 up; K (=H) contiguous
 *   w13_scale  FP32 [E][2I/128][H/128]
 *   w2         E4M3 [E][H][I]   K (=I) contiguous
 *   w2_scale   FP32 [E][H/128][I/128]
 *   out        BF16 [M][H]; rows >= M are never written
 * Numerics: hidden and the activation are quantised per row per 128 columns with
 * scale = amax/448 (1.0 for an all-zero group) and round-to-nearest-even saturating E4M3
 * codes; each GEMM output is sum over 128-blocks kb ascending of P_kb * (sa_kb * sw_kb)
 * in FP32 (P_kb = the block's FP8 dot product on the tensor core or in FP32);
 * act = silu(g) * u in FP32; out = bf16(sum over slots j ascending of w_j * y_j).
 * Up to 256 routed rows the arithmetic is exactly the above. With more (128-row expert
 * tiles) the promotion is one fused multiply-add per block (one rounding instead of two per step), silu's exponential is the
 * hardware base-2 exponential of a split argument with a fast division (a few ulp for every
 * g) and the requantisation multiplies by 448/amax (within one ulp of the division): inside
 * the same tolerances (activation codes may move one step next to a rounding boundary).
 * 0 <= M <= max_tokens; M = 0 is a no-op. */
moe_status_t moe_fp8_forward(const void* hidden, const int32_t* topk_ids, const float* topk_w,
                             int32_t M, const uint8_t* w13, const float* w13_scale,
                             const uint8_t* w2, const float* w2_scale, void* out,
                             void* workspace, size_t workspace_bytes,
                             const moe_fp8_shape_t* shape, cudaStream_t stream);

/* moe_fp8_forward of the RMSNorm'd hidden (see moe_rmsnorm): hidden holds the un-normalised
 * rows; the gate/up kernel (few routed rows) or the quantiser (many) normalises each row as it
 * quantises it. The workspace views qa/sa hold the codes of y. */
moe_status_t moe_fp8_norm_forward(const void* hidden, const void* norm_weight, float eps, const int32_t* topk_ids,
                                  const float* topk_w, int32_t M, const uint8_t* w13, const float* w13_scale,
                                  const uint8_t* w2, const float* w2_scale, void* out, void* workspace,
                                  size_t workspace_bytes, const moe_fp8_shape_t* shape, cudaStream_t stream);

/* Routing and the routed expert FFN in one call: moe_route then moe_fp8_forward, enqueued
 * together (arguments as for those calls; topk_ids / topk_w, device [M][K], receive the
 * routing). Results are those of the two calls. */
moe_status_t moe_fp8_route_forward(const void* hidden, const void* router_w, const float* bias, int32_t M,
                                   int32_t renormalize, const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                   const float* w2_scale, void* out, int32_t* topk_ids, float* topk_w,
                                   void* workspace, size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                   cudaStream_t stream);

/* moe_fp8_route_forward of the RMSNorm'd hidden: moe_norm_route then moe_fp8_norm_forward
 * (three launches at decode, as without the norm). */
moe_status_t moe_fp8_norm_route_forward(const void* hidden, const void* norm_weight, float eps, const void* router_w,
                                        const float* bias, int32_t M, int32_t renormalize, const uint8_t* w13,
                                        const float* w13_scale, const uint8_t* w2, const float* w2_scale, void* out,
                                        int32_t* topk_ids, float* topk_w, void* workspace, size_t workspace_bytes,
                                        const moe_fp8_shape_t* shape, cudaStream_t stream);

/* The same layer as ONE kernel launch ([NK] prefill-pair section: one producer made of
 * semantic routing, gate/up, SiLU and quantisation, down-partial and metadata stages, with
 * the route reducer's fixed reduction order), for a few routed pairs: M * top_k <= 16,
 * M <= 16, E <= 256 and a multiple of 8, inter <= 2048, hidden <= 8192, and the pipeline
 * fitting the device; otherwise MOE_ERR_UNSUPPORTED. Results (routing, output, and the
 * workspace views qa, sa, act, act_scale in pair order) are bitwise those of
 * moe_fp8_route_forward. The work is split into (routed pair, 128-column activation block)
 * units spread over 16-CTA clusters, one CTA per SM: each cluster routes the tokens itself
 * (the router's arithmetic), runs its units' gate/up with the hidden quantisation, SiLU*up and
 * the requantisation, and the down projection's K block of each unit; the last CTA to finish
 * an output block (an arrival counter in the workspace) sums the down terms over K blocks and
 * then slots in ascending order. It is slower than the two calls at decode on GB300 (the
 * whole layer's latency chain sits in one grid, and consecutive launches cannot overlap it);
 * it exists for callers that need the layer as a single launch. The arrival counters are left
 * at zero by every call; after a call that reported MOE_STATUS_WAIT_TIMEOUT, re-initialise the
 * workspace (moe_fp8_workspace_init) before the next call. router_w and bias are read while
 * the previous kernel on `stream` may still run (as for moe_route). */
moe_status_t moe_fp8_route_forward_one_launch(const void* hidden, const void* router_w, const float* bias,
                                              int32_t M, int32_t renormalize, const uint8_t* w13,
                                              const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                              void* out, int32_t* topk_ids, float* topk_w, void* workspace,
                                              size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                              cudaStream_t stream);

/* The speculative-verify layer as the two operations of [NK]'s prefill-pair section: a
 * producer (semantic routing, gate/up, SiLU and quantisation, down partials and metadata) and
 * a route reducer with its own ABI, launch geometry and fixed reduction order. Both carry an
 * exact batch guard ([NK]: a kernel whose grid depends on the batch takes one; the profile
 * compiled here is verify_m12 with one request): M == 12 with hidden 2048, inter 768,
 * 128 experts and top-8, else MOE_ERR_UNSUPPORTED.
 * moe_fp8_verify_produce routes the 12 tokens (ids and weights into topk_ids / topk_w, as
 * moe_route; arguments as for moe_fp8_route_forward) and leaves in the workspace every routed
 * pair's down projection y (FP32, at the row the sort gives it: perm_row[t*8 + j]), the
 * activation codes and scales and the hidden codes (the views of moe_fp8_workspace_view).
 * It runs the router, the quantise-and-sort of moe_fp8_prepare and the expert-grouped
 * gate/up and down kernels (each expert's weights read once for the tokens routed to it).
 * moe_fp8_verify_reduce then writes out[t] = bf16(sum over slots j ascending of
 * topk_w[t][j] * y[perm_row[t*8 + j]]) (FP32 multiply then add, from 0); call it after the
 * producer on the same stream and workspace. produce + reduce equals moe_fp8_route_forward
 * bit for bit, and its arithmetic is that of the pair kernels (moe_fp8_gate_up_direct +
 * moe_fp8_down_combine).
 * moe_fp8_verify_produce_one_launch is the same producer as one launch of 16-CTA clusters
 * (each cluster routes for itself, then takes a share of the distinct routed experts), with
 * the identity permutation and y in pair order; the same reducer follows it. It is opt-in:
 * MOE_ERR_UNSUPPORTED also when the device cannot hold its clusters. */
moe_status_t moe_fp8_verify_produce(const void* hidden, const void* router_w, const float* bias, int32_t M,
                                    int32_t renormalize, const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                    const float* w2_scale, int32_t* topk_ids, float* topk_w, void* workspace,
                                    size_t workspace_bytes, const moe_fp8_shape_t* shape, cudaStream_t stream);
moe_status_t moe_fp8_verify_produce_one_launch(const void* hidden, const void* router_w, const float* bias, int32_t M,
                                               int32_t renormalize, const uint8_t* w13, const float* w13_scale,
                                               const uint8_t* w2, const float* w2_scale, int32_t* topk_ids,
                                               float* topk_w, void* workspace, size_t workspace_bytes,
                                               const moe_fp8_shape_t* shape, cudaStream_t stream);
moe_status_t moe_fp8_verify_reduce(const float* topk_w, int32_t M, void* out, void* workspace, size_t workspace_bytes,
                                   const moe_fp8_shape_t* shape, cudaStream_t stream);

/* The four stages of moe_fp8_forward as separate calls, for callers that interleave them
 * with other work or time them one by one. They communicate through the workspace and
 * must be enqueued in this order on one stream with the same M and shape. */
moe_status_t moe_fp8_prepare(const void* hidden, const int32_t* topk_ids, int32_t M,
                             void* workspace, size_t workspace_bytes,
                             const moe_fp8_shape_t* shape, cudaStream_t stream);
moe_status_t moe_fp8_gate_up(const uint8_t* w13, const float* w13_scale, int32_t M,
                             void* workspace, size_t workspace_bytes,
                             const moe_fp8_shape_t* shape, cudaStream_t stream);
moe_status_t moe_fp8_down(const uint8_t* w2, const float* w2_scale, int32_t M, void* workspace,
                          size_t workspace_bytes, const moe_fp8_shape_t* shape,
                          cudaStream_t stream);
moe_status_t moe_fp8_combine(const float* topk_w, int32_t M, void* out, void* workspace,
                             size_t workspace_bytes, const moe_fp8_shape_t* shape,
                             cudaStream_t stream);

/* The layer split at its expert partials, for callers that move routed rows between devices
 * (expert parallelism: [AMDK] names ranks<n> kernels and sums expert partials in a fixed order
 * "inside the next kernel"; [NK] keeps the route reducer a separate operation).
 * moe_fp8_forward_partials runs moe_fp8_prepare, moe_fp8_gate_up and moe_fp8_down and writes
 * every routed pair's down projection in pair order:
 *   y_out  FP32 [M*K][H], row t*K + j = y of token t's slot j (zeros for a skipped pair)
 * moe_fp8_combine_pairs is the route reducer over such rows (wherever they were computed):
 *   out[t] = bf16(sum over slots j ascending of topk_w[t][j] * y[t*K + j]), FP32 multiply
 *   then add from 0, pairs whose topk_ids entry is outside [0, E) skipped.
 * moe_fp8_combine_pairs(moe_fp8_forward_partials(...)) equals moe_fp8_forward bit for bit;
 * combine_pairs needs no workspace. Other arguments and limits as for moe_fp8_forward. */
moe_status_t moe_fp8_forward_partials(const void* hidden, const int32_t* topk_ids, int32_t M, const uint8_t* w13,
                                      const float* w13_scale, const uint8_t* w2, const float* w2_scale, float* y_out,
                                      void* workspace, size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                      cudaStream_t stream);
moe_status_t moe_fp8_combine_pairs(const float* y, const int32_t* topk_ids, const float* topk_w, int32_t M, void* out,
                                   const moe_fp8_shape_t* shape, cudaStream_t stream);

/* The layer with MXFP4 expert weights ([AMDK] MoE shape token mxfp4_h6144_i768_e128_top4;
 * [NKL] supported-targets table: MXFP4 kernels checked against FP64 dequantised references).
 * Up to 64 routed rows (M * top_k): two launches, one unit per (token, slot) pair -- gate/up
 * quantising hidden itself, then down fused with the combine. Above: quantise and sort the
 * pairs by expert (as moe_fp8_prepare), gate/up and down over groups of up to 16 rows of one
 * expert (each expert's weights read once per group), then the slot-order combine.
 *   hidden, topk_ids, topk_w, out, workspace, shape: as for moe_fp8_forward
 *   w13q       u8 [E][2I][H/2]  E2M1 codes, two per byte, the lower K index in the low nibble
 *                               (rows 0..I-1 gate, I..2I-1 up)
 *   w13_scale  u8 [E][2I][H/32] UE8M0 scale of each 32 consecutive K elements of a row
 *                               (2^(e - 127); e = 255 is NaN)
 *   w2q        u8 [E][H][I/2];  w2_scale u8 [E][H][I/32]
 *   w13q and w2q must be 32-byte aligned (the tensor maps that expand the packed codes for
 *   the tensor core require it), else MOE_ERR_INVALID_ARG.
 * Numerics: hidden and the activation as for moe_fp8_forward (E4M3 per 128 columns); each
 * GEMM output is, per 128-wide K block kb ascending, T_kb = sum over its four 32-wide
 * sub-blocks s ascending of P_s * 2^(e_s - 127) (FP32 from 0; P_s the 32-term dot product of
 * the E4M3 activation and E2M1 weight values, summed in FP32 on the tensor core), then
 * acc = acc + T_kb * sa_kb (FP32 from 0); SiLU, requantisation and the slot-order combine as
 * for moe_fp8_forward. The tensor core reads the E2M1 codes directly (kind::f8f6f4 with an
 * E2M1 operand; every E2M1 value is an E4M3 value, so each product is exact).
 * moe_mxfp4_route_forward is moe_route then moe_mxfp4_forward. */
moe_status_t moe_mxfp4_forward(const void* hidden, const int32_t* topk_ids, const float* topk_w, int32_t M,
                               const uint8_t* w13q, const uint8_t* w13_scale, const uint8_t* w2q,
                               const uint8_t* w2_scale, void* out, void* workspace, size_t workspace_bytes,
                               const moe_fp8_shape_t* shape, cudaStream_t stream);
moe_status_t moe_mxfp4_route_forward(const void* hidden, const void* router_w, const float* bias, int32_t M,
                                     int32_t renormalize, const uint8_t* w13q, const uint8_t* w13_scale,
                                     const uint8_t* w2q, const uint8_t* w2_scale, void* out, int32_t* topk_ids,
                                     float* topk_w, void* workspace, size_t workspace_bytes,
                                     const moe_fp8_shape_t* shape, cudaStream_t stream);

/* moe_mxfp4_forward's path above 64 routed rows as stage calls, between moe_fp8_prepare
 * (quantise and sort) and moe_fp8_combine, all on one stream with the same M and shape:
 * moe_mxfp4_gate_up writes the activation codes and scales at the sorted rows, moe_mxfp4_down
 * the FP32 down projections y at the sorted rows. MOE_ERR_UNSUPPORTED for M * top_k <= 64
 * (moe_fp8_prepare does not sort so few rows). Weights and numerics as moe_mxfp4_forward;
 * prepare + gate_up + down + combine equals moe_mxfp4_forward bit for bit. */
moe_status_t moe_mxfp4_gate_up(const uint8_t* w13q, const uint8_t* w13_scale, int32_t M, void* workspace,
                               size_t workspace_bytes, const moe_fp8_shape_t* shape, cudaStream_t stream);
moe_status_t moe_mxfp4_down(const uint8_t* w2q, const uint8_t* w2_scale, int32_t M, void* workspace,
                            size_t workspace_bytes, const moe_fp8_shape_t* shape, cudaStream_t stream);

/* moe_mxfp4_forward's pair path (up to 256 routed rows) as its two kernels (as
 * moe_fp8_gate_up_direct / moe_fp8_down_combine):
 * moe_mxfp4_gate_up_direct quantises hidden and writes the activation codes and scales in
 * pair order to the workspace; moe_mxfp4_down_combine reads them and writes out. The down
 * call reads topk_ids, topk_w, w2q and w2_scale while the kernel launched before it on
 * `stream` may still be running (that kernel must not write them). Limits and errors as
 * for moe_mxfp4_forward. */
moe_status_t moe_mxfp4_gate_up_direct(const void* hidden, const int32_t* topk_ids, int32_t M, const uint8_t* w13q,
                                      const uint8_t* w13_scale, void* workspace, size_t workspace_bytes,
                                      const moe_fp8_shape_t* shape, cudaStream_t stream);
moe_status_t moe_mxfp4_down_combine(const int32_t* topk_ids, const float* topk_w, int32_t M, const uint8_t* w2q,
                                    const uint8_t* w2_scale, void* out, void* workspace, size_t workspace_bytes,
                                    const moe_fp8_shape_t* shape, cudaStream_t stream);

/* The few-routed-row path as its two kernels (one unit per (token, slot) pair; M * top_k
 * <= 256), the layout of the accepted M=1 MoE objects of [ARCH] (gate/up + SiLU +
 * quantisation, then down/reduce). moe_fp8_forward runs these two kernels when M * top_k
 * <= 64 (its gate/up launch also prefetches the routed experts' w2 blocks into L2; the
 * arithmetic is the same); above that it sorts the pairs by expert, which re-reads fewer
 * weights. MOE_ERR_UNSUPPORTED above 256 rows. moe_fp8_gate_up_direct quantises hidden itself and writes the activation codes
 * and scales (pair order) to the workspace; moe_fp8_down_combine reads them and writes out
 * with the combine of moe_fp8_combine (slot order, FP32 multiply then add, from 0).
 * moe_fp8_down_combine reads topk_ids, topk_w, w2 and w2_scale while the kernel launched
 * just before it on `stream` (normally moe_fp8_gate_up_direct) may still be running, so
 * that kernel must not write them; the activation is read only after it has completed. */
moe_status_t moe_fp8_gate_up_direct(const void* hidden, const int32_t* topk_ids, int32_t M,
                                    const uint8_t* w13, const float* w13_scale, void* workspace,
                                    size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                    cudaStream_t stream);
/* moe_fp8_gate_up_direct as moe_fp8_forward launches it for few routed rows: the same kernel,
 * which also prefetches the routed experts' w2 and w2_scale blocks into L2 once its own
 * weights have landed (so the down launch after it reads them from L2). Outputs equal
 * moe_fp8_gate_up_direct's bit for bit; arguments and limits as for it, plus w2 / w2_scale. */
moe_status_t moe_fp8_gate_up_prefetch(const void* hidden, const int32_t* topk_ids, int32_t M, const uint8_t* w13,
                                      const float* w13_scale, const uint8_t* w2, const float* w2_scale,
                                      void* workspace, size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                      cudaStream_t stream);
moe_status_t moe_fp8_down_combine(const int32_t* topk_ids, const float* topk_w, int32_t M,
                                  const uint8_t* w2, const float* w2_scale, void* out, void* workspace,
                                  size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                  cudaStream_t stream);

/* Debug view of the workspace (device pointers into it, valid after moe_fp8_prepare /
 * moe_fp8_gate_up / moe_fp8_down of the same M): hidden codes qa u8 [M][H], hidden scales
 * sa f32 [M][H/128], expert-sorted routed rows: row_src i32 [R] (flat pair index t*K+j of
 * sorted row r), perm_row i32 [M*K] (sorted row of pair t*K+j, -1 if skipped), act codes
 * u8 [R][I], act scales f32 [R][I/128], y f32 [R][H]; R = M*K. Any out pointer may be
 * NULL. moe_fp8_route_forward_one_launch writes qa, sa (its own quantiser), act and
 * act_scale in pair order (row t*K+j); it writes no permutation and no y. */
typedef struct {
  uint8_t* qa;
  float* sa;
  int32_t* row_src;
  int32_t* perm_row;
  uint8_t* act;
  float* act_scale;
  float* y;
  int32_t* expert_offsets; /* i32 [E+1] start of each expert's rows */
  int32_t* topk_ids;       /* i32 [M][K], f32 [M][K]: the routing of the last */
  float* topk_w;           /*   moe_fp8_route_forward_host call */
  uint32_t* tickets;       /* u32 [min(max_tokens,16)][H/128]: the arrival counters of
                              moe_fp8_route_forward_one_launch (zero between calls) */
} moe_fp8_ws_view_t;
moe_status_t moe_fp8_workspace_view(void* workspace, size_t workspace_bytes,
                                    const moe_fp8_shape_t* shape, moe_fp8_ws_view_t* view);

/* The whole layer for a caller holding the tokens in host memory: one call enqueues on
 * `stream` the copy of hidden to the device (into the workspace), moe_route, moe_fp8_forward
 * and the copy of out back to the host, and returns at once; the caller synchronises the
 * stream before reading host_out. No counterpart in the paper: this is an addition of this
 * library (a host-facing entry for integrations that keep activations in host memory).
 *   host_hidden  BF16 [M][H] host memory, read by the first copy
 *   host_out     BF16 [M][H] host memory, written by the last copy
 *   the other arguments as for moe_route and moe_fp8_forward (router_w, bias, w13, w13_scale,
 *   w2, w2_scale are device pointers).
 * Page-locked (pinned or registered) host buffers are read and written by the kernels
 * directly, without copies. Other host memory goes through device copies in the workspace;
 * with pageable memory the driver stages those copies and the call returns only when they
 * are done. The routing is kept in the workspace (moe_fp8_workspace_view: topk_ids,
 * topk_w). Results equal moe_route then moe_fp8_forward on the same inputs. */
moe_status_t moe_fp8_route_forward_host(const void* host_hidden, void* host_out, int32_t M,
                                        const void* router_w, const float* bias, int32_t renormalize,
                                        const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                        const float* w2_scale, void* workspace, size_t workspace_bytes,
                                        const moe_fp8_shape_t* shape, cudaStream_t stream);

/* moe_fp8_route_forward_host for host buffers the caller guarantees are page-locked and
 * mapped (cudaMallocHost / cudaHostAlloc, or cudaHostRegister on a device that can use host
 * pointers for registered memory): the kernels read host_hidden and write host_out in place
 * through unified addressing, with no pointer-type query and no copy on the call's path.
 * host_hidden and host_out must be 16-byte aligned. Passing pageable memory is a caller
 * error (the kernels' accesses to it fail). No counterpart in the paper (as above). */
moe_status_t moe_fp8_route_forward_pinned(const void* host_hidden, void* host_out, int32_t M,
                                          const void* router_w, const float* bias, int32_t renormalize,
                                          const uint8_t* w13, const float* w13_scale, const uint8_t* w2,
                                          const float* w2_scale, void* workspace, size_t workspace_bytes,
                                          const moe_fp8_shape_t* shape, cudaStream_t stream);

/* moe_fp8_forward for callers that cannot allocate device memory where they run the layer
 * (for example while a memory pool is locked or being resized, inside callbacks that must
 * not enter the allocator, or in integrations without a device allocator): the same
 * arguments as moe_fp8_forward minus the workspace. No counterpart in the paper: this is
 * an addition of this library. The intermediate activation lives in a 1 MiB scratch array
 * compiled into the library (a file-scope __device__ array that every GPU loading the
 * library keeps until process exit), so this call allocates nothing.
 * It runs the kernels of moe_fp8_gate_up_direct + moe_fp8_down_combine.
 * Limits: M * top_k <= 256 and M * top_k * (inter + inter/32) + 512 <= 1 MiB; anything
 * larger returns MOE_ERR_UNSUPPORTED.
 * Set-up: the first call in a CUDA context (made with that context current) looks up the
 * array's device address; make that first call before any stream capture. The address is
 * kept per (device, context) for the life of the process, so a process that calls
 * cudaDeviceReset must not call this entry point on that device again.
 * Sharing: all calls on a device share the array, which keeps the last call's contents;
 * calls whose GPU work overlaps (unordered streams) race on it. Each call clears the
 * array's status word on `stream`; device status bits are not readable through this call.
 * Numerics and outputs are identical to moe_fp8_gate_up_direct + moe_fp8_down_combine, and so
 * to moe_fp8_forward when M * top_k <= 64. */
moe_status_t moe_fp8_forward_noalloc(const void* hidden, const int32_t* topk_ids, const float* topk_w,
                                     int32_t M, const uint8_t* w13, const float* w13_scale,
                                     const uint8_t* w2, const float* w2_scale, void* out,
                                     const moe_fp8_shape_t* shape, cudaStream_t stream);

/* Self-check of the bounded device wait that every kernel uses ([NKL] "Development
 * expectations": a focused correctness entry point per kernel contract). One thread waits on a barrier phase
 * that nothing completes, gives up after limit_us microseconds (1 .. 10^6), sets
 * MOE_STATUS_WAIT_TIMEOUT in the workspace's status word and returns; the context stays
 * usable. Clear the status afterwards with moe_fp8_workspace_init. */
moe_status_t moe_fp8_selftest_wait(void* workspace, size_t workspace_bytes, const moe_fp8_shape_t* shape,
                                   uint32_t limit_us, cudaStream_t stream);

/* Copy the workspace's status word to host memory `host_dst` (asynchronous on `stream`;
 * the caller synchronises before reading it). */
moe_status_t moe_fp8_read_status(const void* workspace, uint32_t* host_dst, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_FP8_H_ */
