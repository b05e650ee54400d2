// oracle.cpp -- plain, slow CPU restatement of the routed FP8 block-scaled MoE FFN.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call this
// file: only the tests, the package's smoke check and the benchmark's CPU-baseline leg
// use it. It shares no code, header, table or constant generator with the CUDA library.
//
// Sources for what is computed (the pages are prose; every numeric detail that they
// leave open is marked "reading"):
//   * "NetraRuntime/netra-kernel" README (older lab README), "Supported targets" table:
//     weights are FP8 E4M3 with one FP32 scale per 128x128 block.
//   * "NetraRuntime/netra-kernel" README, prefill-pair build section: the routed MoE
//     producer is routing -> gate/up -> SiLU and quantisation -> down-partial -> metadata,
//     and a separate route reducer sums the down partials per route in its own fixed order.
//   * docs/compiler/architecture.md, accepted M=1 MoE objects: gate/up, SiLU+quant and
//     down/reduce; intermediates are an FP32 gate/up tensor, an FP8 activation and an
//     activation-scale tensor.
//   * "Inferact/amd-kernels" README, reduction rule: partial sums are added in a fixed
//     order, never with atomic adds.
//   * netra-kernel README, kernel-contract field list: accumulation, rounding and reduction
//     order are part of an operation's identity, so the orders used below are the contract.
//
// Precision: every step is FP32 unless stated; each 128-term FP8 block dot product is
// formed exactly in double and rounded to FP32 once (it is exact: see block_dot()).
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -shared -fPIC (no FMA contraction, so the
// FP32 chains below round exactly where they are written, on x86-64 and on aarch64).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

namespace {

// ---------------------------------------------------------------------------------------
// FP8 E4M3 ("fn" variant) from the format definition: 1 sign bit, 4 exponent bits with
// bias 7, 3 mantissa bits; exponent field 0 is subnormal (m * 2^-9); the all-ones
// exponent with mantissa 7 is NaN (no infinities); the largest finite magnitude is
// 1.75 * 2^8 = 448 (code 0x7E).
// ---------------------------------------------------------------------------------------
float e4m3_value(unsigned code) {
  const unsigned s = (code >> 7) & 1u, ex = (code >> 3) & 15u, m = code & 7u;
  double mag;
  if (ex == 15u && m == 7u) return s ? -NAN : NAN;
  if (ex == 0u) mag = std::ldexp((double)m, -9);                 // subnormal
  else mag = std::ldexp((double)(8u + m), (int)ex - 10);         // (1 + m/8) * 2^(ex-7)
  return (float)(s ? -mag : mag);
}

struct Table {
  float v[256];
  Table() { for (unsigned c = 0; c < 256; ++c) v[c] = e4m3_value(c); }
};
const Table& table() { static Table t; return t; }

// Round-to-nearest-even encoder with saturation to +-448 ("satfinite"): the nearest of the
// 127 non-negative finite magnitudes (codes 0x00..0x7E), ties to the code whose lowest bit
// is 0; magnitudes at or above 448 clamp to 448; NaN stays NaN; the sign bit is kept, so a
// negative value that rounds to zero is 0x80.
uint8_t e4m3_encode(float x) {
  const unsigned sign = std::signbit(x) ? 0x80u : 0u;
  if (std::isnan(x)) return (uint8_t)(sign | 0x7Fu);
  const double a = std::fabs((double)x);
  const float* t = table().v;
  if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);
  unsigned lo = 0;  // largest code with magnitude <= a
  for (unsigned c = 0; c <= 0x7Eu; ++c)
    if ((double)t[c] <= a) lo = c;
  if ((double)t[lo] == a) return (uint8_t)(sign | lo);
  const unsigned hi = lo + 1;  // lo < 0x7E here because a < 448
  const double dlo = a - (double)t[lo], dhi = (double)t[hi] - a;  // exact in double
  unsigned c;
  if (dlo < dhi) c = lo;
  else if (dhi < dlo) c = hi;
  else c = (lo & 1u) ? hi : lo;
  return (uint8_t)(sign | c);
}

float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// FP32 -> BF16, round to nearest even on the bit pattern (NaN kept quiet).
uint16_t f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40u);
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

// Quantiser Q over one group of n values (n = 128: one scale per token per 128 columns).
// Reading: amax/448 is an IEEE FP32 division; an all-zero group takes scale 1.0 so that
// its codes are all zero (the pages do not say what a zero group does).
float quantise_group(const float* v, int n, uint8_t* q) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) amax = std::max(amax, std::fabs(v[i]));
  float s = amax / 448.0f;
  if (amax == 0.0f) s = 1.0f;
  for (int i = 0; i < n; ++i) q[i] = e4m3_encode(v[i] / s);
  return s;
}

// Exact 128-term block dot product of FP8 codes, rounded once to FP32.
// Every E4M3 value is an integer multiple of 2^-9 below 2^18 in units, so each product
// is an integer multiple of 2^-18 below 2^36 units and any sum of 128 of them stays
// below 2^43 units < 2^53: the double accumulation below is exact.
float block_dot(const uint8_t* a, const uint8_t* w, int n) {
  const float* t = table().v;
  double s = 0.0;
  for (int k = 0; k < n; ++k) s += (double)t[a[k]] * (double)t[w[k]];
  return (float)s;
}

struct Dims { int M, H, I, E, K; };

// ---------------------------------------------------------------------------------------
// MXFP4 (OCP microscaling, FP4 elements): E2M1 codes -- 1 sign bit, 2 exponent bits with
// bias 1, 1 mantissa bit; exponent field 0 is subnormal (m * 0.5); no infinities or NaN; the
// largest magnitude is 1.5 * 2^2 = 6 -- with one UE8M0 scale per 32 consecutive elements
// (8 exponent bits, value 2^(e - 127), e = 255 is NaN).
// ---------------------------------------------------------------------------------------
double e2m1_value(unsigned code) {
  const unsigned s = (code >> 3) & 1u, ex = (code >> 1) & 3u, m = code & 1u;
  const double mag = ex == 0u ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, (int)ex - 1);
  return s ? -mag : mag;
}
float ue8m0_value(unsigned e) { return e == 255u ? NAN : (float)std::ldexp(1.0, (int)e - 127); }

// One MXFP4 block-scaled GEMV row (reading for the MXFP4 weight variant): for each 128-wide
// K block kb (the activation's quantisation group),
//   T_kb = sum over its 32-wide sub-blocks s ascending of fl32(P_s) * 2^(e_s - 127),
// with P_s the exact 32-term dot product of the E4M3 activation values and the E2M1 weight
// values, each multiply and add one FP32 operation from 0; then, as for FP8 weights,
//   out = sum over kb ascending of fl32(T_kb * sa[kb]), from 0.
// wq: the row's codes, two per byte, the lower K index in the low nibble; ws: its scales.
// abs_sum receives sum |P_s * 2^e_s * sa| (the error-scale reference of the tests).
float mx_row(const uint8_t* a, const float* sa, const uint8_t* wq, const uint8_t* ws, int nkb, float* abs_sum) {
  const float* t = table().v;
  float acc = 0.0f;
  double asum = 0.0;
  for (int kb = 0; kb < nkb; ++kb) {
    float T = 0.0f;
    for (int j = 0; j < 4; ++j) {
      const int s = kb * 4 + j;
      double d = 0.0;  // exact: multiples of 2^-10 below 2^12 in magnitude, 32 terms
      for (int k = s * 32; k < s * 32 + 32; ++k) {
        const unsigned code = (wq[k / 2] >> (4 * (k & 1))) & 15u;
        d += (double)t[a[k]] * e2m1_value(code);
      }
      const float p = (float)d;
      const float sc = ue8m0_value(ws[s]);
      const float term = p * sc;
      T = T + term;
      asum += std::fabs((double)term * (double)sa[kb]);
    }
    const float term = T * sa[kb];
    acc = acc + term;
  }
  if (abs_sum) *abs_sum = (float)asum;
  return acc;
}

// Down projection of one routed pair with MXFP4 w2: codes [E][H][I/2], scales [E][H][I/32].
void mx_down_row(const uint8_t* qact, const float* s2, int e, const Dims d, const uint8_t* w2q, const uint8_t* w2s,
                 float* y) {
  const int H = d.H, I = d.I;
  for (int h = 0; h < H; ++h) {
    const int64_t row = (int64_t)e * H + h;
    y[h] = mx_row(qact, s2, w2q + row * (I / 2), w2s + row * (I / 32), I / 128, nullptr);
  }
}

}  // namespace

extern "C" {

// ---- codec ---------------------------------------------------------------------------
void orc_e4m3_table(float* out256) { for (int c = 0; c < 256; ++c) out256[c] = table().v[c]; }

void orc_e4m3_encode(const float* x, uint8_t* q, int64_t n) {
  for (int64_t i = 0; i < n; ++i) q[i] = e4m3_encode(x[i]);
}

// Q over consecutive groups of `group` values: q[n], s[n/group].
void orc_quantise(const float* x, int64_t n, int group, uint8_t* q, float* s) {
  for (int64_t g = 0; g < n / group; ++g) s[g] = quantise_group(x + g * group, group, q + g * group);
}

void orc_bf16_round(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(x[i]);
}

// Exact block dot product, exposed for the block-sum pin.
float orc_block_dot(const uint8_t* a, const uint8_t* w, int n) { return block_dot(a, w, n); }

// ---- RMS normalisation ---------------------------------------------------------------
// RMSNorm of the hidden rows ahead of the layer (netra-kernel lab README, repository layout:
// gfx950 "normalization and quantization fusions"; the model's RMSNorm in front of the MoE
// block). The pages give no epsilon and no weight convention; reading: the plain definition
//   y[k] = bf16_rn( (x[k] * r) * gamma[k] ),   r = 1 / sqrt(ss / H + eps),
// with eps and gamma (BF16 [H]) supplied by the caller, and ss = the sum of x[k]^2 formed like
// the router's logits: an FP32 fma chain over each 128-wide chunk (k ascending, from 0), the
// chunks added in ascending order. Every step is one correctly rounded FP32 operation: the
// division by H, the add of eps, the square root, the reciprocal (1 / s as a division), and
// the two multiplies. x and y are BF16 [M][H]; rstd_out [M] (optional) receives r.
int orc_rmsnorm(const uint16_t* x, const uint16_t* gamma, float eps, int M, int H, uint16_t* y, float* rstd_out) {
  if (M < 0 || H <= 0 || H % 128) return -1;
  for (int t = 0; t < M; ++t) {
    const uint16_t* xr = x + (int64_t)t * H;
    float ss = 0.0f;
    for (int c = 0; c < H / 128; ++c) {
      float acc = 0.0f;
      for (int k = c * 128; k < c * 128 + 128; ++k) {
        const float v = bf16_to_f32(xr[k]);
        acc = std::fmaf(v, v, acc);
      }
      ss = ss + acc;
    }
    const float mean = ss / (float)H;
    const float s = std::sqrt(mean + eps);
    const float r = 1.0f / s;
    if (rstd_out) rstd_out[t] = r;
    for (int k = 0; k < H; ++k) {
      const float v = (bf16_to_f32(xr[k]) * r) * bf16_to_f32(gamma[k]);
      y[(int64_t)t * H + k] = f32_to_bf16(v);
    }
  }
  return 0;
}

// ---- routing -------------------------------------------------------------------------
// Router (netra-kernel README capability table: BF16 routing; prefill-pair section:
// "semantic routing" stage). hidden BF16 [M][H] row-major, router_w BF16 [H][E] (E
// contiguous), optional FP32 bias [E].
//   Reading (accumulation order is contract): logit[t][e] = sum over 128-wide chunks c,
//   ascending, of acc_c, where acc_c is an FP32 fused multiply-add chain over the chunk's
//   k ascending, starting at 0. The BF16 x BF16 products are exact in FP32, so fma and
//   mul-then-add agree inside a chunk. The bias is added after the sum.
//   Selection: logits descending, ties to the lower expert index, first K.
//   Weights (renormalize != 0): softmax over the K selected logits; (renormalize == 0):
//   the full softmax over all E, read at the selected experts. Evaluated in double from
//   the FP32 logits and rounded once.
// logits_out [M][E] is optional (NULL to skip). Returns 0, or -1 on bad sizes.
int orc_route(const uint16_t* hidden, const uint16_t* router_w, const float* bias, int M, int H,
              int E, int K, int renormalize, int32_t* ids, float* weights, float* logits_out) {
  if (M < 0 || H <= 0 || H % 128 || E <= 0 || K <= 0 || K > E) return -1;
  std::vector<float> logit(E);
  std::vector<char> taken(E);
  for (int t = 0; t < M; ++t) {
    for (int e = 0; e < E; ++e) {
      float l = 0.0f;
      for (int c = 0; c < H / 128; ++c) {
        float acc = 0.0f;
        for (int k = c * 128; k < c * 128 + 128; ++k)
          acc = std::fmaf(bf16_to_f32(hidden[(int64_t)t * H + k]),
                          bf16_to_f32(router_w[(int64_t)k * E + e]), acc);
        l = l + acc;
      }
      if (bias) l = l + bias[e];
      logit[e] = l;
      if (logits_out) logits_out[(int64_t)t * E + e] = l;
    }
    std::fill(taken.begin(), taken.end(), 0);
    for (int j = 0; j < K; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || logit[e] > logit[best])) best = e;
      taken[best] = 1;
      ids[(int64_t)t * K + j] = best;
    }
    const double lmax = (double)logit[ids[(int64_t)t * K]];
    double den = 0.0;
    if (renormalize) {
      for (int j = 0; j < K; ++j) den += std::exp((double)logit[ids[(int64_t)t * K + j]] - lmax);
    } else {
      for (int e = 0; e < E; ++e) den += std::exp((double)logit[e] - lmax);
    }
    for (int j = 0; j < K; ++j)
      weights[(int64_t)t * K + j] =
          (float)(std::exp((double)logit[ids[(int64_t)t * K + j]] - lmax) / den);
  }
  return 0;
}

// ---- expert FFN and combine -----------------------------------------------------------
// Optional intermediates of orc_moe_forward (any pointer may be NULL).
typedef struct {
  uint8_t* qa;      // [M][H]      hidden codes
  float* sa;        // [M][H/128]  hidden scales
  float* g;         // [M][K][I]   gate pre-activation (FP32 promotion chain result)
  float* u;         // [M][K][I]   up pre-activation
  float* gabs;      // [M][K][I]   sum over blocks of |P * scale| for g (error-scale reference)
  float* uabs;      // [M][K][I]   same for u
  float* act;       // [M][K][I]   silu(g) * u before quantisation
  uint8_t* qact;    // [M][K][I]   activation codes
  float* s2;        // [M][K][I/128] activation scales
  float* y;         // [M][K][H]   down projection of each routed pair
} orc_debug_t;

namespace {

// One block-scaled GEMV row: out = sum over 128-blocks kb ascending of
//   fl32(exact block dot) * fl32(sa[kb] * sw[kb]),
// each product and sum a separate FP32 operation starting from 0 (reading: the order
// "scale product, multiply, add" is this library's contract; the pages fix only that
// block scales apply per 128-K slice to FP32 partials).
float scaled_row(const uint8_t* a, const float* sa, const uint8_t* w, const float* sw_row,
                 int nkb, float* abs_sum) {
  float acc = 0.0f;
  double asum = 0.0;
  for (int kb = 0; kb < nkb; ++kb) {
    const float p = block_dot(a + kb * 128, w + kb * 128, 128);
    const float sc = sa[kb] * sw_row[kb];
    const float term = p * sc;
    acc = acc + term;
    asum += std::fabs((double)term);
  }
  if (abs_sum) *abs_sum = (float)asum;
  return acc;
}

// Down projection of one routed pair (step 6): y[h] for every row h of w2[e] ([H][I], K
// contiguous), from the pair's activation codes and scales.
void down_row(const uint8_t* qact, const float* s2, int e, const Dims d, const uint8_t* w2, const float* s2w,
              float* y) {
  const int H = d.H, I = d.I, nki = I / 128;
  for (int h = 0; h < H; ++h) {
    const uint8_t* wrow = w2 + ((int64_t)e * H + h) * I;
    const float* srow = s2w + ((int64_t)e * (H / 128) + h / 128) * nki;
    y[h] = scaled_row(qact, s2, wrow, srow, nki, nullptr);
  }
}

// Combine (step 7, the route reducer): slots j ascending, FP32 multiply then add, from 0;
// a skipped slot contributes nothing; BF16 round to nearest even.
void combine_token(const float* Y, const float* w_t, const char* valid, int K, int H, uint16_t* out_t) {
  for (int h = 0; h < H; ++h) {
    float acc = 0.0f;
    for (int j = 0; j < K; ++j) {
      if (!valid[j]) continue;
      const float p = w_t[j] * Y[(size_t)j * H + h];
      acc = acc + p;
    }
    out_t[h] = f32_to_bf16(acc);
  }
}

void forward_tokens(const uint16_t* hidden, const int32_t* ids, const float* w, const Dims d,
                    const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2w,
                    uint16_t* out, const orc_debug_t* dbg, int t0, int t1) {
  const int M = d.M, H = d.H, I = d.I, E = d.E, K = d.K;
  (void)M;
  const int nkh = H / 128, nki = I / 128;
  std::vector<float> x(H), sa(nkh), G(2 * I), Gabs(2 * I), act(I), s2(nki), Y((size_t)K * H);
  std::vector<uint8_t> qa(H), qact(I);
  std::vector<char> valid(K);
  for (int t = t0; t < t1; ++t) {
    for (int k = 0; k < H; ++k) x[k] = bf16_to_f32(hidden[(int64_t)t * H + k]);
    for (int kb = 0; kb < nkh; ++kb) sa[kb] = quantise_group(&x[kb * 128], 128, &qa[kb * 128]);
    if (dbg && dbg->qa) std::memcpy(dbg->qa + (int64_t)t * H, qa.data(), H);
    if (dbg && dbg->sa) std::memcpy(dbg->sa + (int64_t)t * nkh, sa.data(), nkh * 4);
    for (int j = 0; j < K; ++j) {
      const int e = ids[(int64_t)t * K + j];
      valid[j] = (e >= 0 && e < E);
      if (!valid[j]) continue;  // reading: an out-of-range id contributes nothing
      const int64_t pj = (int64_t)t * K + j;
      // gate/up: rows n of w13[e] ([2I][H], K contiguous); gate = n < I, up = n >= I
      for (int n = 0; n < 2 * I; ++n) {
        const uint8_t* wrow = w13 + ((int64_t)e * 2 * I + n) * H;
        const float* srow = s13 + ((int64_t)e * (2 * I / 128) + n / 128) * nkh;
        G[n] = scaled_row(qa.data(), sa.data(), wrow, srow, nkh, &Gabs[n]);
      }
      // SiLU(gate) * up, evaluated in double from the FP32 g, u and rounded once
      for (int i = 0; i < I; ++i) {
        const double g = G[i], u = G[I + i];
        act[i] = (float)(g / (1.0 + std::exp(-g)) * u);
      }
      for (int kb = 0; kb < nki; ++kb) s2[kb] = quantise_group(&act[kb * 128], 128, &qact[kb * 128]);
      float* y = &Y[(size_t)j * H];
      down_row(qact.data(), s2.data(), e, d, w2, s2w, y);
      if (dbg) {
        if (dbg->g) std::memcpy(dbg->g + pj * I, G.data(), I * 4);
        if (dbg->u) std::memcpy(dbg->u + pj * I, G.data() + I, I * 4);
        if (dbg->gabs) std::memcpy(dbg->gabs + pj * I, Gabs.data(), I * 4);
        if (dbg->uabs) std::memcpy(dbg->uabs + pj * I, Gabs.data() + I, I * 4);
        if (dbg->act) std::memcpy(dbg->act + pj * I, act.data(), I * 4);
        if (dbg->qact) std::memcpy(dbg->qact + pj * I, qact.data(), I);
        if (dbg->s2) std::memcpy(dbg->s2 + pj * nki, s2.data(), nki * 4);
        if (dbg->y) std::memcpy(dbg->y + pj * H, y, (size_t)H * 4);
      }
    }
    combine_token(Y.data(), w + (int64_t)t * K, valid.data(), K, H, out + (int64_t)t * H);
  }
}

// The MXFP4 forward for tokens [t0, t1): the FP8 steps with MXFP4 weight rows (mx_row).
void mx_forward_tokens(const uint16_t* hidden, const int32_t* ids, const float* w, const Dims d,
                       const uint8_t* w13q, const uint8_t* w13s, const uint8_t* w2q, const uint8_t* w2s,
                       uint16_t* out, const orc_debug_t* dbg, int t0, int t1) {
  const int H = d.H, I = d.I, E = d.E, K = d.K;
  const int nkh = H / 128, nki = I / 128;
  std::vector<float> x(H), sa(nkh), G(2 * I), Gabs(2 * I), act(I), s2(nki), Y((size_t)K * H);
  std::vector<uint8_t> qa(H), qact(I);
  std::vector<char> valid(K);
  for (int t = t0; t < t1; ++t) {
    for (int k = 0; k < H; ++k) x[k] = bf16_to_f32(hidden[(int64_t)t * H + k]);
    for (int kb = 0; kb < nkh; ++kb) sa[kb] = quantise_group(&x[kb * 128], 128, &qa[kb * 128]);
    if (dbg && dbg->qa) std::memcpy(dbg->qa + (int64_t)t * H, qa.data(), H);
    if (dbg && dbg->sa) std::memcpy(dbg->sa + (int64_t)t * nkh, sa.data(), nkh * 4);
    for (int j = 0; j < K; ++j) {
      const int e = ids[(int64_t)t * K + j];
      valid[j] = (e >= 0 && e < E);
      if (!valid[j]) continue;
      const int64_t pj = (int64_t)t * K + j;
      for (int n = 0; n < 2 * I; ++n) {
        const int64_t row = (int64_t)e * 2 * I + n;
        G[n] = mx_row(qa.data(), sa.data(), w13q + row * (H / 2), w13s + row * (H / 32), nkh, &Gabs[n]);
      }
      for (int i = 0; i < I; ++i) {
        const double g = G[i], u = G[I + i];
        act[i] = (float)(g / (1.0 + std::exp(-g)) * u);
      }
      for (int kb = 0; kb < nki; ++kb) s2[kb] = quantise_group(&act[kb * 128], 128, &qact[kb * 128]);
      float* y = &Y[(size_t)j * H];
      mx_down_row(qact.data(), s2.data(), e, d, w2q, w2s, y);
      if (dbg) {
        if (dbg->g) std::memcpy(dbg->g + pj * I, G.data(), I * 4);
        if (dbg->u) std::memcpy(dbg->u + pj * I, G.data() + I, I * 4);
        if (dbg->gabs) std::memcpy(dbg->gabs + pj * I, Gabs.data(), I * 4);
        if (dbg->uabs) std::memcpy(dbg->uabs + pj * I, Gabs.data() + I, I * 4);
        if (dbg->act) std::memcpy(dbg->act + pj * I, act.data(), I * 4);
        if (dbg->qact) std::memcpy(dbg->qact + pj * I, qact.data(), I);
        if (dbg->s2) std::memcpy(dbg->s2 + pj * nki, s2.data(), nki * 4);
        if (dbg->y) std::memcpy(dbg->y + pj * H, y, (size_t)H * 4);
      }
    }
    combine_token(Y.data(), w + (int64_t)t * K, valid.data(), K, H, out + (int64_t)t * H);
  }
}

void mx_down_combine_tokens(const uint8_t* qact, const float* s2, const int32_t* ids, const float* w, const Dims d,
                            const uint8_t* w2q, const uint8_t* w2s, uint16_t* out, int t0, int t1) {
  const int H = d.H, I = d.I, E = d.E, K = d.K, nki = I / 128;
  std::vector<float> Y((size_t)K * H);
  std::vector<char> valid(K);
  for (int t = t0; t < t1; ++t) {
    for (int j = 0; j < K; ++j) {
      const int e = ids[(int64_t)t * K + j];
      valid[j] = (e >= 0 && e < E);
      if (!valid[j]) continue;
      const int64_t pj = (int64_t)t * K + j;
      mx_down_row(qact + pj * I, s2 + pj * nki, e, d, w2q, w2s, &Y[(size_t)j * H]);
    }
    combine_token(Y.data(), w + (int64_t)t * K, valid.data(), K, H, out + (int64_t)t * H);
  }
}

// Steps 6 and 7 for M tokens from given activation codes and scales (per routed pair).
void down_combine_tokens(const uint8_t* qact, const float* s2, const int32_t* ids, const float* w, const Dims d,
                         const uint8_t* w2, const float* s2w, uint16_t* out, int t0, int t1) {
  const int H = d.H, I = d.I, E = d.E, K = d.K, nki = I / 128;
  std::vector<float> Y((size_t)K * H);
  std::vector<char> valid(K);
  for (int t = t0; t < t1; ++t) {
    for (int j = 0; j < K; ++j) {
      const int e = ids[(int64_t)t * K + j];
      valid[j] = (e >= 0 && e < E);
      if (!valid[j]) continue;
      const int64_t pj = (int64_t)t * K + j;
      down_row(qact + pj * I, s2 + pj * nki, e, d, w2, s2w, &Y[(size_t)j * H]);
    }
    combine_token(Y.data(), w + (int64_t)t * K, valid.data(), K, H, out + (int64_t)t * H);
  }
}

}  // namespace

// The whole FFN for M tokens: quantise hidden per token per 128 columns, for each routed
// pair (t, j) with e = ids[t][j] compute the gate/up rows, SiLU(g)*u, requantise per 128
// columns, the down rows, then combine the K pairs of each token in slot order into BF16.
// Layouts: hidden BF16 [M][H]; ids int32 [M][K]; w FP32 [M][K]; w13 E4M3 [E][2I][H];
// s13 FP32 [E][2I/128][H/128]; w2 E4M3 [E][H][I]; s2w FP32 [E][H/128][I/128];
// out BF16 [M][H]. `nthreads` > 1 splits the tokens over std::threads (timing only: the
// per-token arithmetic is identical). Returns 0, or -1 on bad sizes.
int orc_moe_forward(const uint16_t* hidden, const int32_t* ids, const float* w, int M, int H,
                    int I, int E, int K, const uint8_t* w13, const float* s13, const uint8_t* w2,
                    const float* s2w, uint16_t* out, const orc_debug_t* dbg, int nthreads) {
  if (M < 0 || H <= 0 || I <= 0 || H % 128 || I % 128 || E <= 0 || K <= 0) return -1;
  const Dims d{M, H, I, E, K};
  table();  // build the decode table before any thread starts
  if (nthreads <= 1 || M <= 1) {
    forward_tokens(hidden, ids, w, d, w13, s13, w2, s2w, out, dbg, 0, M);
    return 0;
  }
  nthreads = std::min(nthreads, M);
  std::vector<std::thread> th;
  for (int i = 0; i < nthreads; ++i) {
    const int t0 = (int)((int64_t)M * i / nthreads), t1 = (int)((int64_t)M * (i + 1) / nthreads);
    th.emplace_back(forward_tokens, hidden, ids, w, d, w13, s13, w2, s2w, out, dbg, t0, t1);
  }
  for (auto& x : th) x.join();
  return 0;
}

// Steps 6 and 7 alone: the down projection of every routed pair from GIVEN activation
// codes qact [M][K][I] and scales s2 [M][K][I/128], then the slot-order combine into BF16
// out [M][H] -- the same arithmetic as the tail of orc_moe_forward, so that the output of
// a path whose activation codes are known can be checked on its own. Returns 0 or -1.
int orc_down_combine(const uint8_t* qact, const float* s2, const int32_t* ids, const float* w, int M, int H,
                     int I, int E, int K, const uint8_t* w2, const float* s2w, uint16_t* out, int nthreads) {
  if (M < 0 || H <= 0 || I <= 0 || H % 128 || I % 128 || E <= 0 || K <= 0) return -1;
  const Dims d{M, H, I, E, K};
  table();
  if (nthreads <= 1 || M <= 1) {
    down_combine_tokens(qact, s2, ids, w, d, w2, s2w, out, 0, M);
    return 0;
  }
  nthreads = std::min(nthreads, M);
  std::vector<std::thread> th;
  for (int i = 0; i < nthreads; ++i) {
    const int t0 = (int)((int64_t)M * i / nthreads), t1 = (int)((int64_t)M * (i + 1) / nthreads);
    th.emplace_back(down_combine_tokens, qact, s2, ids, w, d, w2, s2w, out, t0, t1);
  }
  for (auto& x : th) x.join();
  return 0;
}

// ---- MXFP4 weight variant --------------------------------------------------------------
void orc_e2m1_table(float* out16) { for (unsigned c = 0; c < 16; ++c) out16[c] = (float)e2m1_value(c); }
void orc_ue8m0_decode(const uint8_t* e, float* out, int64_t n) { for (int64_t i = 0; i < n; ++i) out[i] = ue8m0_value(e[i]); }
float orc_mx_row(const uint8_t* a, const float* sa, const uint8_t* wq, const uint8_t* ws, int nkb) {
  return mx_row(a, sa, wq, ws, nkb, nullptr);
}

// The FFN of orc_moe_forward with MXFP4 expert weights: w13q u8 [E][2I][H/2] and w13s u8
// [E][2I][H/32]; w2q u8 [E][H][I/2] and w2s u8 [E][H][I/32] (codes two per byte, lower K
// index in the low nibble; one UE8M0 scale per 32 elements along K). Activations, SiLU, the
// requantisation and the combine are those of the FP8 layer. Returns 0 or -1.
int orc_mxfp4_forward(const uint16_t* hidden, const int32_t* ids, const float* w, int M, int H, int I, int E, int K,
                      const uint8_t* w13q, const uint8_t* w13s, const uint8_t* w2q, const uint8_t* w2s,
                      uint16_t* out, const orc_debug_t* dbg, int nthreads) {
  if (M < 0 || H <= 0 || I <= 0 || H % 128 || I % 128 || E <= 0 || K <= 0) return -1;
  const Dims d{M, H, I, E, K};
  table();
  if (nthreads <= 1 || M <= 1) {
    mx_forward_tokens(hidden, ids, w, d, w13q, w13s, w2q, w2s, out, dbg, 0, M);
    return 0;
  }
  nthreads = std::min(nthreads, M);
  std::vector<std::thread> th;
  for (int i = 0; i < nthreads; ++i) {
    const int t0 = (int)((int64_t)M * i / nthreads), t1 = (int)((int64_t)M * (i + 1) / nthreads);
    th.emplace_back(mx_forward_tokens, hidden, ids, w, d, w13q, w13s, w2q, w2s, out, dbg, t0, t1);
  }
  for (auto& x : th) x.join();
  return 0;
}

// orc_down_combine with MXFP4 w2.
int orc_mxfp4_down_combine(const uint8_t* qact, const float* s2, const int32_t* ids, const float* w, int M, int H,
                           int I, int E, int K, const uint8_t* w2q, const uint8_t* w2s, uint16_t* out, int nthreads) {
  if (M < 0 || H <= 0 || I <= 0 || H % 128 || I % 128 || E <= 0 || K <= 0) return -1;
  const Dims d{M, H, I, E, K};
  table();
  if (nthreads <= 1 || M <= 1) {
    mx_down_combine_tokens(qact, s2, ids, w, d, w2q, w2s, out, 0, M);
    return 0;
  }
  nthreads = std::min(nthreads, M);
  std::vector<std::thread> th;
  for (int i = 0; i < nthreads; ++i) {
    const int t0 = (int)((int64_t)M * i / nthreads), t1 = (int)((int64_t)M * (i + 1) / nthreads);
    th.emplace_back(mx_down_combine_tokens, qact, s2, ids, w, d, w2q, w2s, out, t0, t1);
  }
  for (auto& x : th) x.join();
  return 0;
}

}  // extern "C"
