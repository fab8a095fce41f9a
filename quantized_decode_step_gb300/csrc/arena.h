// Activation arena planner (host): lifetime intervals -> byte offsets.
#pragma once
#include <stdint.h>

#include <string>
#include <vector>

namespace mag {

struct ArenaTensor {
  std::string name;
  uint64_t size;   // bytes
  int first;       // producer op index
  int last;        // last consumer op index (closed interval)
  uint64_t offset; // planned
};

// Greedy by size ("TFLite memory planner" 2.2): tensors largest first (ties:
// earlier first op, then lower index), each at the lowest `align`-multiple
// offset that overlaps no already placed tensor whose closed lifetime
// [first, last] meets its own ("TFLite memory planner" 2.1: a tensor lives
// from its producer to its last consumer, and an op reads its inputs while it
// writes its output). no_reuse gives every tensor its own bytes (the
// preserve-all debug mode of "TFLite memory planner" 3.2). Returns the arena
// size, a multiple of `align`.
uint64_t plan_arena(std::vector<ArenaTensor>& tensors, uint64_t align, bool no_reuse);

}  // namespace mag
