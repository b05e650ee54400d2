// Host-only client of the pair-kernel launch planner (csrc/pair_plan.h), built and run by
// tests/test_plan_host.py with the host C++ compiler: no CUDA, no GPU. For each case it
// prints the plan and the facts the test checks it against, one line per case:
//   sms smem_per_sm mode nkb units K split nst smem_total resident
#include <cstdio>

#include "pair_plan.h"

using namespace moe;

template <int MODE>
void show(const PlanDevice& d, int nkb, long long units, int K, bool allow_split, int fixed_cluster) {
  const PairPlan p = plan_pair<MODE>(d, nkb, units, K, allow_split, fixed_cluster);
  const size_t smem = pair_smem<MODE>(p.nst, nkb / p.split, K).total;
  const int cluster = fixed_cluster ? fixed_cluster : p.split;
  std::printf("%d %zu %d %d %lld %d %d %d %zu %lld\n", d.sms, d.smem_per_sm, MODE, nkb, units, K, p.split, p.nst,
              smem, (long long)resident_ctas(d, cluster, smem));
}

// MXFP4 pair kernels: mode 10 = gate/up, 11 = down fused with the combine (cluster of K)
template <bool GATEUP>
void show_mx(const PlanDevice& d, int nkb, long long units, int K) {
  const PairPlan p = plan_mx<GATEUP>(d, nkb, units, K);
  const size_t smem = mx_request<GATEUP>(d, p.nst, nkb / p.split, K);
  const int cluster = GATEUP ? p.split : K;
  std::printf("%d %zu %d %d %lld %d %d %d %zu %lld\n", d.sms, d.smem_per_sm, GATEUP ? 10 : 11, nkb, units, K, p.split,
              p.nst, smem, (long long)resident_ctas(d, cluster, smem));
}

int main() {
  const PlanDevice devs[] = {{152, 233472, 232448}, {148, 233472, 232448}, {132, 233472, 232448},
                             {76, 233472, 232448}, {38, 233472, 232448}, {8, 233472, 232448},
                             {152, 102400, 101376}};
  for (const PlanDevice& d : devs) {
    // decode gate/up (h2048: 16 K blocks, 8 pairs x 6 output blocks), verify (96 pairs),
    // wide (h6144: 48 K blocks, 4 pairs x 6), down+combine (6 K blocks, cluster of K)
    show<kGateUpFused>(d, 16, 48, 8, true, 0);
    show<kGateUpFused>(d, 16, 576, 8, true, 0);
    show<kGateUpFused>(d, 48, 24, 4, true, 0);
    show<kGateUpWs>(d, 16, 48, 8, true, 0);
    show<kDownY>(d, 6, 128, 8, true, 0);
    show<kDownCombine>(d, 6, 16, 8, false, 8);
    show<kDownCombine>(d, 6, 192, 8, false, 8);
    // MXFP4 h6144/i768/top4: decode (4 pairs x 6 blocks), 64 tokens (256 pairs); down + combine
    show_mx<true>(d, 48, 24, 4);
    show_mx<true>(d, 48, 1536, 4);
    show_mx<true>(d, 2, 8, 2);
    show_mx<false>(d, 6, 48, 4);
    show_mx<false>(d, 6, 3072, 4);
  }
  return 0;
}
