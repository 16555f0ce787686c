// jfa_bbs_plan: Base Batch Shuffling, the data-parallel batch balancer.
//
// Meta GEM MFU write-up (piletech.kr/articles/112134), details section, Base Batch
// Shuffling bullet: 128-sample sub-batches are sorted by sequence length and the
// heaviest and the lightest are merged in turn, which evens out the work of the GPUs
// without any all-to-all between ranks.  The pages give no more than that; the plan
// below is the plainest reading (the readings are listed with the declaration in
// include/jfa.h):
//   1. the global batch is cut into consecutive sub-batches of `sub` samples;
//   2. a sub-batch costs the sum of its samples' costs;
//   3. sub-batches are sorted heaviest first (ties by index);
//   4. the i-th heaviest is merged with the i-th lightest into pair i (the middle one
//      stays single when the count is odd);
//   5. pairs go to ranks in serpentine order (0, 1, .., R-1, R-1, .., 0, 0, 1, ..), so
//      each rank receives the same number of pairs, within one.
// Every rank computes the same plan from the per-sample costs (lengths are known to
// every rank's loader) and then loads only its own samples: no data crosses ranks.
// Host code only; nothing here touches a GPU.
#include <stdint.h>

#include <algorithm>
#include <numeric>
#include <vector>

#include "internal.h"

extern "C" jfa_status jfa_bbs_plan(const int64_t* cost, int64_t n_samples, int32_t sub, int32_t ranks,
                                   int32_t* sub_rank, int32_t* sub_slot, int64_t* rank_cost) {
  if (n_samples < 0 || sub < 1 || ranks < 1) return JFA_ERR_INVALID_ARG;
  const int64_t n_sub = (n_samples + sub - 1) / sub;
  if (n_sub > INT32_MAX) return JFA_ERR_INVALID_ARG;
  if (n_samples > 0 && (cost == nullptr || sub_rank == nullptr || sub_slot == nullptr))
    return JFA_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n_samples; ++i)
    if (cost[i] < 0) return JFA_ERR_INVALID_ARG;

  // 1-2. sub-batch costs
  std::vector<int64_t> sc((size_t)n_sub, 0);
  for (int64_t i = 0; i < n_samples; ++i) sc[(size_t)(i / sub)] += cost[i];
  // 3. heaviest first, ties by index
  std::vector<int32_t> order((size_t)n_sub);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return sc[a] > sc[b]; });
  // 4-5. pair i = (i-th heaviest, i-th lightest); pairs to ranks in serpentine order
  std::vector<int32_t> filled((size_t)ranks, 0);
  if (rank_cost != nullptr)
    for (int32_t r = 0; r < ranks; ++r) rank_cost[r] = 0;
  const int64_t n_pairs = (n_sub + 1) / 2;
  for (int64_t p = 0; p < n_pairs; ++p) {
    const int64_t round = p / ranks, k = p % ranks;
    const int32_t r = (int32_t)((round & 1) ? ranks - 1 - k : k);
    const int32_t heavy = order[(size_t)p], light = order[(size_t)(n_sub - 1 - p)];
    sub_rank[heavy] = r;
    sub_slot[heavy] = filled[r]++;
    if (rank_cost != nullptr) rank_cost[r] += sc[heavy];
    if (light != heavy) {
      sub_rank[light] = r;
      sub_slot[light] = filled[r]++;
      if (rank_cost != nullptr) rank_cost[r] += sc[light];
    }
  }
  return JFA_OK;
}
