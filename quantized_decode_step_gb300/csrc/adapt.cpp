// Load profile and plan / pool policies; see adapt.h.
#include "adapt.h"

#include <algorithm>
#include <cmath>

#include "mag.h"

namespace mag {

LoadProfile::LoadProfile(int window, int sample_every)
    : window_(std::max(1, window)), sample_every_(std::max(1, sample_every)) {
  ring_.reserve(window_);
}

bool LoadProfile::observe(int32_t length) {
  const bool take = seen_ % sample_every_ == 0;
  ++seen_;
  if (!take) return false;
  if ((int)ring_.size() < window_) {
    ring_.push_back(length);
  } else {
    ring_[head_] = length;
    head_ = (head_ + 1) % window_;
  }
  return true;
}

int32_t LoadProfile::quantile(double q) const {
  const int n = (int)ring_.size();
  if (n == 0) return -1;
  std::vector<int32_t> v(ring_);
  std::sort(v.begin(), v.end());
  // rank ceil(q n), computed in integers for q given to 1e-9 (avoids 0.9 * 64 = 57.6000...01 -> 58)
  const int64_t qn = (int64_t)std::llround(q * 1e9) * n;
  int64_t rank = (qn + 999999999) / 1000000000;
  rank = std::min<int64_t>(std::max<int64_t>(rank, 1), n);
  return v[rank - 1];
}

int plan_for(int32_t p90, int32_t short_below, int32_t long_above) {
  if (p90 < short_below) return 0;
  if (p90 > long_above) return 2;
  return 1;
}

int64_t hot_pool_blocks(int32_t p90, int32_t n_sessions, double slack, int block_tokens) {
  if (p90 <= 0 || n_sessions <= 0) return 0;
  const int64_t x = (int64_t)n_sessions * ((p90 + block_tokens - 1) / block_tokens);
  // slack x, rounded up, with slack taken to six decimals (a float 1.2 is 1.20000005: in binary the
  // product 1.2 x 10 would round up to 13)
  const int64_t micro = std::llround(slack * 1e6);
  return (micro * x + 999999) / 1000000;
}

}  // namespace mag

// ---------------------------------------------------------------- C ABI: the profile on its own
struct mag_profiler {
  mag::LoadProfile p;
};

extern "C" {

mag_status mag_profiler_create(int32_t window, int32_t sample_every, mag_profiler** out) {
  if (!out) return MAG_ERR_INVALID_ARG;
  *out = nullptr;
  if (window < 1 || sample_every < 1) return MAG_ERR_INVALID_ARG;
  *out = new mag_profiler{mag::LoadProfile(window, sample_every)};
  return MAG_OK;
}

void mag_profiler_destroy(mag_profiler* p) { delete p; }

int32_t mag_profiler_observe(mag_profiler* p, int32_t length) { return p && p->p.observe(length) ? 1 : 0; }

mag_status mag_profiler_quantile(const mag_profiler* p, double q, int32_t* out) {
  if (!p || !out || !(q > 0.0 && q <= 1.0)) return MAG_ERR_INVALID_ARG;
  *out = p->p.quantile(q);
  return MAG_OK;
}

int32_t mag_profiler_count(const mag_profiler* p) { return p ? p->p.count() : 0; }

int32_t mag_plan_for(int32_t p90, int32_t short_below, int32_t long_above) {
  return mag::plan_for(p90, short_below, long_above);
}

int64_t mag_hot_pool_blocks(int32_t p90, int32_t n_sessions, float slack) {
  return mag::hot_pool_blocks(p90, n_sessions, slack, 16);
}

}  // extern "C"
