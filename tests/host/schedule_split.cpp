// Host check of the logits work split: the schedule header's cost model and item
// iteration, compiled for the CPU.  For random groups (rows, longest context) and grid
// sizes, every CTA's items (first from the cost range's first group on, as the start
// record and the kernel's iterator take them) must cover every tile of every group
// exactly once, in increasing order.  Prints "OK <cases>" or the first failure.
#define __host__
#define __device__
#define __forceinline__ inline
#include "../../sparse_attention_fp4_gb300/csrc/schedule.cuh"

#include <cstdio>
#include <cstdlib>
#include <random>
#include <vector>

using namespace fp4idx;

int main(int argc, char** argv) {
  const unsigned seed = argc > 1 ? (unsigned)atoi(argv[1]) : 1u;
  const int cases = argc > 2 ? atoi(argv[2]) : 300;
  std::mt19937 rng(seed);
  for (int cs = 0; cs < cases; cs++) {
    const int n_groups = (int)(rng() % 300);
    const int num_ctas = 1 + (int)(rng() % 400);
    std::vector<int32_t> row0(n_groups + 1), maxlen(n_groups), seq(n_groups);
    std::vector<int64_t> prefix(n_groups + 1);
    row0[0] = 0;
    prefix[0] = 0;
    for (int g = 0; g < n_groups; g++) {
      const int rows = 1 + (int)(rng() % kGroupMax);
      const int kind = (int)(rng() % 8);
      maxlen[g] = kind == 0 ? 0 : kind == 1 ? 1 + (int)(rng() % 200) : (int)(rng() % 70000);
      seq[g] = g;
      row0[g + 1] = row0[g] + rows;
      prefix[g + 1] = prefix[g] + group_cost(maxlen[g], rows);
    }
    const int64_t W = prefix[n_groups];
    std::vector<std::vector<int>> claimed(n_groups);
    for (int g = 0; g < n_groups; g++) claimed[g].assign((maxlen[g] + kTileTokens - 1) / kTileTokens, 0);
    auto r0a = [&](int32_t i) { return row0[i]; };
    auto mla = [&](int32_t i) { return maxlen[i]; };
    auto sqa = [&](int32_t i) { return seq[i]; };
    auto pra = [&](int32_t i) { return prefix[i]; };
    for (int c = 0; c < num_ctas; c++) {
      const int64_t lo = W * c / num_ctas, hi = W * (c + 1) / num_ctas;
      int32_t g = first_group_after(prefix.data(), n_groups, lo);
      Item it;
      int32_t last_g = -1;
      while (next_item(r0a, mla, sqa, pra, n_groups, lo, hi, g, it)) {
        if (it.g <= last_g || it.t0 >= it.t1 || it.t0 < 0 || it.t1 > (int)claimed[it.g].size() ||
            it.r0 != row0[it.g] || it.rows != row0[it.g + 1] - row0[it.g] || it.maxlen != maxlen[it.g] ||
            it.seq != seq[it.g]) {
          printf("FAIL case %d cta %d: bad item g=%d [%d,%d)\n", cs, c, it.g, it.t0, it.t1);
          return 1;
        }
        last_g = it.g;
        for (int t = it.t0; t < it.t1; t++) claimed[it.g][t]++;
      }
    }
    for (int g = 0; g < n_groups; g++)
      for (size_t t = 0; t < claimed[g].size(); t++)
        if (claimed[g][t] != 1) {
          printf("FAIL case %d: group %d tile %zu claimed %d times\n", cs, g, t, claimed[g][t]);
          return 1;
        }
  }
  printf("OK %d\n", cases);
  return 0;
}
