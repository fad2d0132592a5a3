// Host planning of the backward kernel's static schedule (see bwd_item).
#include <algorithm>
#include <cstring>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <utility>
#include <vector>

#include "fattn_sched.h"

namespace fattn {

namespace {

constexpr int kTile = 128;

// Costs in half Q tiles: a K/V tile walking n Q tiles costs 2n + 1 (the 1 is
// the item's own start-up and dK/dV write-out, about half a step), so a pair
// costs 2 (n_tiles + 1) + 2.
long long pair_cost(int n_tiles) { return 2LL * (n_tiles + 1) + 2; }
long long single_cost(int n_tiles, int j) { return 2LL * (n_tiles - j) + 1; }

// Pairs that the snake deal of n_paired pairs gives CTA c of G (as bwd_item).
int pairs_of(int n_paired, int G, int c) {
  const int rounds = n_paired / G;
  const int pos = (rounds & 1) ? (G - 1 - c) : c;
  return rounds + (pos < n_paired - rounds * G ? 1 : 0);
}

// Deals the single K/V tiles of the last `heads` heads after the pairs of the
// others: heaviest first (j ascending, heads inner), each to the CTA with the
// least work so far (the lowest index among equals) -- the longest-
// processing-time-first rule.  Returns the largest CTA cost; fills `lists`
// (one entry list per CTA, in dealing order) when given.
long long deal_tail(int n_tiles, int BH, int heads, int G,
                    std::vector<std::vector<uint16_t>>* lists) {
  using Load = std::pair<long long, int>;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> free_first;
  const int n_paired = (n_tiles / 2) * (BH - heads);
  long long worst = 0;
  for (int c = 0; c < G; ++c) {
    const long long l = pairs_of(n_paired, G, c) * pair_cost(n_tiles);
    free_first.push({l, c});
    worst = std::max(worst, l);
  }
  for (int j = 0; j < n_tiles; ++j) {
    for (int r = 0; r < heads; ++r) {
      Load top = free_first.top();
      free_first.pop();
      top.first += single_cost(n_tiles, j);
      worst = std::max(worst, top.first);
      if (lists) (*lists)[top.second].push_back(static_cast<uint16_t>(r * n_tiles + j));
      free_first.push(top);
    }
  }
  return worst;
}

struct TailPlan {
  int heads = 0;
  std::vector<uint16_t> off;   // G + 1 entries
  std::vector<uint16_t> item;
};

// The number of unpaired heads (at most max_heads) that minimises the most
// loaded CTA, with its tables; no tail when none beats whole pairs.
TailPlan plan_tail(int n_tiles, int BH, int G, int max_heads) {
  TailPlan plan;
  long long best = deal_tail(n_tiles, BH, 0, G, nullptr);
  for (int h = 1; h <= max_heads; ++h) {
    const long long cost = deal_tail(n_tiles, BH, h, G, nullptr);
    if (cost < best) {
      best = cost;
      plan.heads = h;
    }
  }
  plan.off.assign(G + 1, 0);
  if (plan.heads == 0) return plan;
  std::vector<std::vector<uint16_t>> lists(G);
  deal_tail(n_tiles, BH, plan.heads, G, &lists);
  for (int c = 0; c < G; ++c) {
    plan.off[c + 1] = static_cast<uint16_t>(plan.off[c] + lists[c].size());
    plan.item.insert(plan.item.end(), lists[c].begin(), lists[c].end());
  }
  return plan;
}

// Plans depend only on the shape and the grid; the search costs up to a few
// milliseconds, so each is made once per process.
const TailPlan& cached_tail(int n_tiles, int BH, int G, int max_heads) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int>, TailPlan> plans;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(n_tiles, BH, G, max_heads);
  auto it = plans.find(key);
  if (it == plans.end()) it = plans.emplace(key, plan_tail(n_tiles, BH, G, max_heads)).first;
  return it->second;
}

}  // namespace

void plan_bwd_schedule(BwdArgs& a, int n_tiles, int hd, bool causal, bool ordered, int grid,
                       long long l2_bytes) {
  // Heads per section: a third of L2 over what one head's steps keep
  // re-reading (fp32 dQ accumulator, Q, dO, L, D).  Not with the ordered
  // reduction: there the items of a head wait on each other at every Q tile,
  // and the more of them run at once the longer the chains (measured on
  // GB300: 1.8x slower).  Causal items are paired first (equal weights), or
  // keep the all-heads heaviest-first order when n_tiles is odd.
  a.sec_heads = a.BH;
  a.paired = causal && !ordered && (n_tiles % 2) == 0 ? 1 : 0;
  a.tail_heads = 0;
  std::memset(a.tail_off, 0, sizeof(a.tail_off));
  if ((!causal || a.paired) && !ordered) {
    const long long per_head =
        static_cast<long long>(n_tiles) * kTile * (hd * 4 + 2 * hd * 2 + 2 * 4);
    const long long fit = per_head > 0 ? (l2_bytes / 3) / per_head : 1;
    a.sec_heads = static_cast<int>(fit < 1 ? 1 : (fit > a.BH ? a.BH : fit));
  }
  // The unpaired heads run together at the end, as one more section: at most
  // two sections' worth, so that they and the last paired section share L2.
  if (a.paired && grid >= 1 && grid <= kBwdTailMaxCtas) {
    const int max_heads =
        std::min({a.BH, kBwdTailCap / n_tiles, 2 * a.sec_heads});
    if (max_heads >= 1) {
      const TailPlan& plan = cached_tail(n_tiles, a.BH, grid, max_heads);
      a.tail_heads = plan.heads;
      std::copy(plan.off.begin(), plan.off.end(), a.tail_off);
      std::copy(plan.item.begin(), plan.item.end(), a.tail_item);
    }
  }
}

}  // namespace fattn
