#include "arena.h"

#include <algorithm>
#include <numeric>

namespace mag {

static uint64_t round_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

uint64_t plan_arena(std::vector<ArenaTensor>& ts, uint64_t align, bool no_reuse) {
  const size_t n = ts.size();
  std::vector<size_t> order(n);
  std::iota(order.begin(), order.end(), size_t(0));
  std::stable_sort(order.begin(), order.end(), [&](size_t a, size_t b) {
    if (ts[a].size != ts[b].size) return ts[a].size > ts[b].size;
    if (ts[a].first != ts[b].first) return ts[a].first < ts[b].first;
    return a < b;
  });
  std::vector<size_t> placed;
  uint64_t end = 0;
  for (size_t idx : order) {
    ArenaTensor& t = ts[idx];
    if (no_reuse) {
      t.offset = round_up(end, align);
      end = t.offset + t.size;
      placed.push_back(idx);
      continue;
    }
    // placed tensors alive at some op where t is alive, by (offset, end)
    std::vector<size_t> live;
    for (size_t p : placed)
      if (ts[p].first <= t.last && t.first <= ts[p].last) live.push_back(p);
    std::sort(live.begin(), live.end(), [&](size_t a, size_t b) {
      if (ts[a].offset != ts[b].offset) return ts[a].offset < ts[b].offset;
      return ts[a].offset + ts[a].size < ts[b].offset + ts[b].size;
    });
    uint64_t cursor = 0;
    for (size_t p : live) {
      if (round_up(cursor, align) + t.size <= ts[p].offset) break;  // fits in the gap below p
      cursor = std::max(cursor, ts[p].offset + ts[p].size);
    }
    t.offset = round_up(cursor, align);
    end = std::max(end, t.offset + t.size);
    placed.push_back(idx);
  }
  return round_up(end, align);
}

}  // namespace mag
