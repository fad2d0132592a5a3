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

// Work units of one head: n_units units, unit u walking n_tiles - step * u
// Q tiles when causal (step = 1: single K/V tiles; step = 2: the CTA-pair
// kernel's units of two K/V tiles).
struct Units {
  int n_units, n_tiles, step;
  int walk(int u) const { return n_tiles - step * u; }
};

// Costs in half Q tiles: a unit walking n Q tiles costs 2n + 1 (the 1 is the
// item's own start-up and dK/dV write-out, about half a step); a pair of
// units u and n_units - 1 - u, which walk the same total for every u, costs
// the sum plus 2.
long long pair_cost(const Units& m) { return 2LL * (m.walk(0) + m.walk(m.n_units - 1)) + 2; }
long long single_cost(const Units& m, int u) { return 2LL * m.walk(u) + 1; }

// Pairs that the snake deal of n_paired pairs gives CTA c of G (as bwd_item).
int pairs_of(int n_paired, int G, int c) {
  const int rounds = n_paired / G;
  const int pos = (rounds & 1) ? (G - 1 - c) : c;
  return rounds + (pos < n_paired - rounds * G ? 1 : 0);
}

// Deals the single units of the last `heads` heads after the pairs of the
// others: heaviest first (u ascending, heads inner), each to the CTA (or
// cluster) with the least work so far (the lowest index among equals) -- the
// longest-processing-time-first rule.  Returns the largest cost; fills
// `lists` (one entry list per CTA, in dealing order) when given.
long long deal_tail(const Units& um, int BH, int heads, int G,
                    std::vector<std::vector<uint16_t>>* lists) {
  using Load = std::pair<long long, int>;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> free_first;
  const int n_paired = (um.n_units / 2) * (BH - heads);
  long long worst = 0;
  for (int c = 0; c < G; ++c) {
    const long long l = pairs_of(n_paired, G, c) * pair_cost(um);
    free_first.push({l, c});
    worst = std::max(worst, l);
  }
  for (int u = 0; u < um.n_units; ++u) {
    for (int r = 0; r < heads; ++r) {
      Load top = free_first.top();
      free_first.pop();
      top.first += single_cost(um, u);
      worst = std::max(worst, top.first);
      if (lists) (*lists)[top.second].push_back(static_cast<uint16_t>(r * um.n_units + u));
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
TailPlan plan_tail(const Units& um, int BH, int G, int max_heads) {
  TailPlan plan;
  long long best = deal_tail(um, BH, 0, G, nullptr);
  for (int h = 1; h <= max_heads; ++h) {
    const long long cost = deal_tail(um, BH, h, G, nullptr);
    if (cost < best) {
      best = cost;
      plan.heads = h;
    }
  }
  plan.off.assign(G + 1, 0);
  if (plan.heads == 0) return plan;
  std::vector<std::vector<uint16_t>> lists(G);
  deal_tail(um, BH, plan.heads, G, &lists);
  for (int c = 0; c < G; ++c) {
    plan.off[c + 1] = static_cast<uint16_t>(plan.off[c] + lists[c].size());
    plan.item.insert(plan.item.end(), lists[c].begin(), lists[c].end());
  }
  return plan;
}

// Plans depend only on the shape and the grid; the search costs up to a few
// milliseconds, so each is made once per process.
const TailPlan& cached_tail(const Units& um, int BH, int G, int max_heads) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int, int>, TailPlan> plans;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(um.n_units, um.n_tiles, um.step, BH, G, max_heads);
  auto it = plans.find(key);
  if (it == plans.end()) it = plans.emplace(key, plan_tail(um, BH, G, max_heads)).first;
  return it->second;
}

// Heads per section: a third of L2 over what one head's steps keep
// re-reading (fp32 dQ accumulator, Q, dO, L, D).
int section_heads(int BH, int n_tiles, int hd, long long l2_bytes) {
  const long long per_head = static_cast<long long>(n_tiles) * kTile * (hd * 4 + 2 * hd * 2 + 2 * 4);
  const long long fit = per_head > 0 ? (l2_bytes / 3) / per_head : 1;
  return static_cast<int>(fit < 1 ? 1 : (fit > BH ? BH : fit));
}

void fill_tail(BwdArgs& a, const Units& um, int grid) {
  if (a.paired && grid >= 1 && grid <= kBwdTailMaxCtas) {
    const int max_heads = std::min({a.BH, kBwdTailCap / um.n_units, 2 * a.sec_heads});
    if (max_heads >= 1) {
      const TailPlan& plan = cached_tail(um, a.BH, grid, max_heads);
      a.tail_heads = plan.heads;
      std::copy(plan.off.begin(), plan.off.end(), a.tail_off);
      std::copy(plan.item.begin(), plan.item.end(), a.tail_item);
    }
  }
}

}  // namespace

void plan_bwd_schedule(BwdArgs& a, int n_tiles, int hd, bool causal, bool ordered, int grid,
                       long long l2_bytes) {
  // Head sections are not used with the ordered reduction: there the items
  // of a head wait on each other at every Q tile, and the more of them run
  // at once the longer the chains (measured on GB300: 1.8x slower).  Causal
  // items are paired first (equal weights), or keep the all-heads
  // heaviest-first order when n_tiles is odd.
  a.sec_heads = a.BH;
  a.paired = causal && !ordered && (n_tiles % 2) == 0 ? 1 : 0;
  a.tail_heads = 0;
  std::memset(a.tail_off, 0, sizeof(a.tail_off));
  if ((!causal || a.paired) && !ordered) a.sec_heads = section_heads(a.BH, n_tiles, hd, l2_bytes);
  // The unpaired heads run together at the end, as one more section: at most
  // two sections' worth, so that they and the last paired section share L2.
  fill_tail(a, Units{n_tiles, n_tiles, 1}, grid);
}

void plan_bwd2_schedule(BwdArgs& a, int n_tiles, bool causal, int clusters, long long l2_bytes) {
  const int n_units = (n_tiles + 1) / 2;
  a.sec_heads = a.BH;
  a.paired = causal && (n_units % 2) == 0 ? 1 : 0;
  a.tail_heads = 0;
  std::memset(a.tail_off, 0, sizeof(a.tail_off));
  if (!causal || a.paired) a.sec_heads = section_heads(a.BH, n_tiles, 128, l2_bytes);
  fill_tail(a, Units{n_units, n_tiles, 2}, clusters);
}

}  // namespace fattn
