// Host-side work schedules for the persistent kernels (forward, backward).
//
// Every persistent kernel processes a list of independent units (a block of
// query rows of one head, or a block of keys of one KV head).  Under a causal
// mask their costs differ by up to the number of tiles per head, so the order
// in which the workers take them decides both the balance (the busiest worker
// sets the launch time) and which heads' K/V (or Q/dO) tiles are streamed at
// the same time.  The kernels' built-in snake order balances well but starts
// the longest unit of every head at once, so every head's tiles compete for
// L2 and are re-read from DRAM.  The schedule built here visits the heads in
// groups whose tiles fit in L2 and, inside a group, gives the longest units
// first to whichever worker the cost model predicts to be free first: the
// balance of list scheduling with the locality of a head-major order.
#include <algorithm>
#include <cstring>
#include <memory>
#include <mutex>
#include <queue>
#include <vector>

#include "fa_internal.h"

namespace fa {

int sched_group_heads(double bytes_per_head) {
  if (!(bytes_per_head > 0.0)) return 1 << 30;
  const double g = kSchedGroupBytes / bytes_per_head;
  return g < 1.0 ? 1 : (g > 1e9 ? 1 << 30 : static_cast<int>(g));
}

namespace {

struct Entry {
  long long key[12];
  std::unique_ptr<SchedTable> table;
};

std::mutex g_mu;
std::vector<Entry> g_cache;
constexpr size_t kCacheEntries = 32;

// List scheduling of the units, group by group (a group is unit.group /
// merge), longest first within a group; returns the predicted makespan.
double list_schedule(const std::vector<SchedUnit>& info, int workers, int merge,
                     std::vector<std::vector<uint16_t>>* lists) {
  const int units = static_cast<int>(info.size());
  std::vector<int> order(static_cast<size_t>(units));
  for (int u = 0; u < units; ++u) order[static_cast<size_t>(u)] = u;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    const SchedUnit& x = info[static_cast<size_t>(a)];
    const SchedUnit& y = info[static_cast<size_t>(b)];
    if (x.group / merge != y.group / merge) return x.group / merge < y.group / merge;
    return x.cost > y.cost;
  });
  // Min-heap of (predicted free time, worker); ties go to the lower worker.
  using Slot = std::pair<double, int>;
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
  for (int w = 0; w < workers; ++w) free_at.push(Slot(0.0, w));
  lists->assign(static_cast<size_t>(workers), std::vector<uint16_t>());
  double makespan = 0.0;
  for (int u : order) {
    Slot s = free_at.top();
    free_at.pop();
    (*lists)[static_cast<size_t>(s.second)].push_back(static_cast<uint16_t>(u));
    s.first += static_cast<double>(info[static_cast<size_t>(u)].cost);
    makespan = std::max(makespan, s.first);
    free_at.push(s);
  }
  return makespan;
}

// Predicted makespan of the kernels' built-in snake order.
double snake_makespan(const std::vector<SchedUnit>& info, int workers) {
  const int units = static_cast<int>(info.size());
  double worst = 0.0;
  for (int w = 0; w < workers; ++w) {
    double t = 0.0;
    for (int k = 0; k * workers < units; ++k) {
      const int u = k * workers + ((k & 1) ? (workers - 1 - w) : w);
      if (u < units) t += static_cast<double>(info[static_cast<size_t>(u)].cost);
    }
    worst = std::max(worst, t);
  }
  return worst;
}

// Picks the smallest head groups whose schedule is predicted within 0.5% of
// the best balance available (the snake order, or one list over all heads):
// when single units are long against a worker's share, small groups would
// leave the last group's longest units to start late.
bool compute(int workers, int units, void (*describe)(const void*, int, SchedUnit*), const void* ctx,
             SchedTable* t) {
  std::vector<SchedUnit> info(static_cast<size_t>(units));
  int max_group = 0;
  for (int u = 0; u < units; ++u) {
    describe(ctx, u, &info[static_cast<size_t>(u)]);
    max_group = std::max(max_group, info[static_cast<size_t>(u)].group);
  }
  std::vector<std::vector<uint16_t>> lists, best;
  const double whole = list_schedule(info, workers, max_group + 1, &best);
  const double snake = snake_makespan(info, workers);
  const double target = 1.005 * std::min(whole, snake);
  bool found = whole <= target;
  for (int merge = 1; merge <= max_group; merge *= 2) {
    if (list_schedule(info, workers, merge, &lists) <= target) {
      best.swap(lists);
      found = true;
      break;
    }
  }
  if (!found) return false;  // the snake order is best: no table
  int pos = 0;
  for (int w = 0; w < workers; ++w) {
    t->start[w] = static_cast<uint16_t>(pos);
    for (uint16_t u : best[static_cast<size_t>(w)]) t->unit[pos++] = u;
  }
  t->start[workers] = static_cast<uint16_t>(pos);
  t->workers = workers;
  return pos == units;
}

}  // namespace

bool build_schedule(const long long (&key)[12], int workers, int units, void (*describe)(const void*, int, SchedUnit*),
                    const void* ctx, SchedTable* out) {
  out->workers = 0;
  if (workers <= 0 || workers > kSchedMaxWorkers || units <= 0 || units > kSchedCap) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  for (const Entry& e : g_cache) {
    if (std::memcmp(e.key, key, sizeof(e.key)) == 0) {
      std::memcpy(out, e.table.get(), sizeof(SchedTable));
      return out->workers > 0;
    }
  }
  std::unique_ptr<SchedTable> t(new SchedTable);
  std::memset(t.get(), 0, sizeof(SchedTable));
  if (!compute(workers, units, describe, ctx, t.get())) t->workers = 0;
  std::memcpy(out, t.get(), sizeof(SchedTable));
  if (g_cache.size() >= kCacheEntries) g_cache.clear();
  Entry e;
  std::memcpy(e.key, key, sizeof(e.key));
  e.table = std::move(t);
  g_cache.push_back(std::move(e));
  return out->workers > 0;
}

}  // namespace fa
