// Load profile and the policies it drives: the plan bucket of the decode step and the hot size of the
// KV block pool ("Magnitude" 2.1-2.2 and 3.1-3.3: a sliding window of recent inferences, sampled, whose
// P50 / P90 / P99 lengths pick one of three preset plans and size the resident pool). Host code only.
#pragma once
#include <stdint.h>

#include <vector>

namespace mag {

// Sliding window of sampled lengths. One observation in `sample_every` is recorded (the first, then
// every sample_every-th after it); the window keeps the last `window` recorded ones.
class LoadProfile {
 public:
  LoadProfile(int window, int sample_every);
  // Offer one observation; returns true when it was recorded.
  bool observe(int32_t length);
  // Nearest-rank quantile of the recorded lengths in the window: the ceil(q n)-th smallest (q in (0, 1]).
  // -1 while the window is empty.
  int32_t quantile(double q) const;
  int count() const { return (int)ring_.size(); }
  bool full() const { return (int)ring_.size() == window_; }
  int64_t seen() const { return seen_; }
  int window() const { return window_; }
  int sample_every() const { return sample_every_; }

 private:
  int window_, sample_every_;
  int64_t seen_ = 0;
  int head_ = 0;                 // next slot to overwrite once full
  std::vector<int32_t> ring_;    // recorded lengths, at most window_
};

// Plan bucket of a P90 length: 0 (short) below short_below, 2 (long) above long_above, else 1.
int plan_for(int32_t p90, int32_t short_below, int32_t long_above);

// Hot pool size in blocks: slack x the blocks that n_sessions sessions of the P90 length hold
// (ceil(p90 / block_tokens) each), rounded up.
int64_t hot_pool_blocks(int32_t p90, int32_t n_sessions, double slack, int block_tokens);

}  // namespace mag
