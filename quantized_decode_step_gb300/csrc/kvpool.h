// The KV block pool's memory and free list ("5. Core modules" 5.2 preallocated block pool; "Magnitude"
// 2.2 layer 1 and 3.2, the hot / cold pool).
//
// Layout either way: (layer * P + block) * block_bytes from one base address, so the kernels see one
// fixed geometry.
//  * Fixed: one allocation of L x P blocks, zeroed at create; blocks handed out first-in first-out in a
//    caller-given order.
//  * Elastic: the L x P blocks are a reserved virtual range; physical memory is mapped in groups of G
//    blocks (G x block_bytes a multiple of the mapping granularity, in every layer's range), zeroed
//    when mapped. The lowest groups up to the hot size stay mapped (the hot pool); a group above it is
//    mapped when the free blocks run out and released once it is wholly free again and the stream has
//    passed its last use (the cold pool). Free blocks are handed out lowest id first, so high groups
//    drain.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <deque>
#include <functional>
#include <set>
#include <string>
#include <vector>

#include "mag.h"

namespace mag {

class KvPool {
 public:
  KvPool() = default;
  KvPool(const KvPool&) = delete;
  KvPool& operator=(const KvPool&) = delete;
  ~KvPool();

  mag_status init_fixed(int layers, int64_t blocks, int64_t block_bytes, const int32_t* order, cudaStream_t s);
  // `blocks` is rounded up to whole groups; one group is mapped (the initial hot pool).
  mag_status init_elastic(int layers, int64_t blocks, int64_t block_bytes, int device, cudaStream_t s);

  uint8_t* base() const { return base_; }
  int64_t blocks() const { return P_; }
  size_t reserved_bytes() const { return (size_t)L_ * P_ * bb_; }
  bool elastic() const { return elastic_; }
  int64_t group_blocks() const { return elastic_ ? G_ : P_; }

  // Blocks free and mapped now, and blocks a session could still get (with the groups not mapped).
  int64_t free_now() const { return elastic_ ? (int64_t)free_set_.size() : (int64_t)fifo_.size(); }
  int64_t available() const;
  // Make n blocks free and mapped (mapping groups, zeroed on s). KV_FULL leaves everything unchanged.
  mag_status reserve(int64_t n, cudaStream_t s);
  int32_t pop();  // requires free_now() > 0
  void push(int32_t b);

  // Elastic: hot size in blocks (whole groups, at least one): groups below it are mapped now, free
  // groups above it start their release. No-op for a fixed pool.
  mag_status set_hot(int64_t blocks, cudaStream_t s, const std::function<bool(int64_t)>& referenced = nullptr);
  // Elastic: release the free groups above the hot size (each after an event recorded on s now) and
  // unmap those whose event has completed. `referenced(g)`, when given, is asked before a group's release
  // starts: a group some session still lists is kept (and reported as an internal error).
  mag_status trim(cudaStream_t s, const std::function<bool(int64_t)>& referenced = nullptr);

  int64_t hot_blocks() const { return elastic_ ? hot_groups_ * G_ : P_; }
  int64_t mapped_blocks() const;
  size_t mapped_bytes() const { return (size_t)mapped_blocks() * L_ * bb_; }
  // Elastic: whether block b lies in a mapped group (a fixed pool: always).
  bool is_mapped(int32_t b) const;

  std::string err;

 private:
  enum : uint8_t { kUnmapped = 0, kMapped = 1, kReleasing = 2 };
  mag_status map_group(int64_t g, cudaStream_t s);
  mag_status unmap_group(int64_t g);
  void revive(int64_t g);

  bool elastic_ = false;
  int L_ = 0;
  int64_t P_ = 0, bb_ = 0, G_ = 0, n_groups_ = 0, hot_groups_ = 0;
  uint8_t* base_ = nullptr;
  int device_ = 0;
  // fixed
  std::deque<int32_t> fifo_;
  // elastic
  std::set<int32_t> free_set_;
  std::vector<uint8_t> state_;
  std::vector<int64_t> used_;
  std::vector<std::vector<unsigned long long>> handles_;  // per group, one physical allocation per layer
  std::vector<cudaEvent_t> release_ev_;
};

}  // namespace mag
