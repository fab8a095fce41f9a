// KV block pool memory and free list; see kvpool.h.
#include "kvpool.h"

#include "alloc.h"

#include <cuda.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

namespace mag {
namespace {

// Virtual-memory calls of the driver, looked up once through the runtime (no link against libcuda).
struct Vmm {
  decltype(&::cuMemGetAllocationGranularity) granularity = nullptr;
  decltype(&::cuMemAddressReserve) reserve = nullptr;
  decltype(&::cuMemAddressFree) free = nullptr;
  decltype(&::cuMemCreate) create = nullptr;
  decltype(&::cuMemRelease) release = nullptr;
  decltype(&::cuMemMap) map = nullptr;
  decltype(&::cuMemUnmap) unmap = nullptr;
  decltype(&::cuMemSetAccess) access = nullptr;
  bool ok = false;
};

const Vmm& vmm() {
  static Vmm v;
  static std::once_flag once;
  std::call_once(once, [] {
    auto get = [](const char* name, void** fn) {
      cudaDriverEntryPointQueryResult q;
      return cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
             q == cudaDriverEntryPointSuccess && *fn;
    };
    v.ok = get("cuMemGetAllocationGranularity", reinterpret_cast<void**>(&v.granularity)) &&
           get("cuMemAddressReserve", reinterpret_cast<void**>(&v.reserve)) &&
           get("cuMemAddressFree", reinterpret_cast<void**>(&v.free)) &&
           get("cuMemCreate", reinterpret_cast<void**>(&v.create)) &&
           get("cuMemRelease", reinterpret_cast<void**>(&v.release)) &&
           get("cuMemMap", reinterpret_cast<void**>(&v.map)) &&
           get("cuMemUnmap", reinterpret_cast<void**>(&v.unmap)) &&
           get("cuMemSetAccess", reinterpret_cast<void**>(&v.access));
  });
  return v;
}

int64_t gcd64(int64_t a, int64_t b) {
  while (b) {
    const int64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

CUmemAllocationProp device_prop(int device) {
  CUmemAllocationProp p = {};
  p.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  p.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  p.location.id = device;
  return p;
}

}  // namespace

KvPool::~KvPool() {
  if (!elastic_) {
    cudaFree(base_);
    return;
  }
  // the owner has synchronised the stream: every group can go
  for (int64_t g = 0; g < n_groups_; ++g) {
    if (state_[g] != kUnmapped) unmap_group(g);
    if (release_ev_[g]) cudaEventDestroy(release_ev_[g]);
  }
  if (base_) vmm().free((CUdeviceptr)base_, reserved_bytes());
}

mag_status KvPool::init_fixed(int layers, int64_t blocks, int64_t block_bytes, const int32_t* order,
                              cudaStream_t s) {
  L_ = layers;
  P_ = blocks;
  bb_ = block_bytes;
  const size_t bytes = reserved_bytes();
  cudaError_t e = dev_malloc(&base_, bytes);
  if (e != cudaSuccess) {
    err = std::string("KV pool: cudaMalloc: ") + cudaGetErrorString(e);
    base_ = nullptr;
    return MAG_ERR_OOM;
  }
  // zeroed: slots past a session's length read as finite zeros
  if ((e = cudaMemsetAsync(base_, 0, bytes, s)) != cudaSuccess) {
    err = std::string("KV pool: memset: ") + cudaGetErrorString(e);
    return MAG_ERR_CUDA;
  }
  for (int64_t i = 0; i < P_; ++i) fifo_.push_back(order ? order[i] : (int32_t)i);
  return MAG_OK;
}

mag_status KvPool::init_elastic(int layers, int64_t blocks, int64_t block_bytes, int device, cudaStream_t s) {
  const Vmm& v = vmm();
  if (!v.ok) {
    err = "KV pool: the driver's virtual-memory calls are not available";
    return MAG_ERR_UNSUPPORTED;
  }
  elastic_ = true;
  L_ = layers;
  bb_ = block_bytes;
  device_ = device;
  const CUmemAllocationProp prop = device_prop(device);
  size_t gran = 0;
  if (v.granularity(&gran, &prop, CU_MEM_ALLOC_GRANULARITY_MINIMUM) != CUDA_SUCCESS || gran == 0) {
    err = "KV pool: no allocation granularity";
    return MAG_ERR_CUDA;
  }
  // G blocks per group: the least count whose bytes are a whole number of granules
  G_ = (int64_t)gran / gcd64(bb_, (int64_t)gran);
  n_groups_ = (blocks + G_ - 1) / G_;
  P_ = n_groups_ * G_;
  if (P_ > INT32_MAX) {
    err = "KV pool: too many blocks";
    return MAG_ERR_INVALID_ARG;
  }
  CUdeviceptr va = 0;
  if (v.reserve(&va, reserved_bytes(), gran, 0, 0) != CUDA_SUCCESS) {
    err = "KV pool: cuMemAddressReserve failed";
    return MAG_ERR_OOM;
  }
  base_ = reinterpret_cast<uint8_t*>(va);
  state_.assign(n_groups_, kUnmapped);
  used_.assign(n_groups_, 0);
  handles_.assign(n_groups_, {});
  release_ev_.assign(n_groups_, nullptr);
  hot_groups_ = 1;
  return map_group(0, s);
}

mag_status KvPool::map_group(int64_t g, cudaStream_t s) {
  const Vmm& v = vmm();
  const CUmemAllocationProp prop = device_prop(device_);
  const size_t gbytes = (size_t)G_ * bb_;
  std::vector<unsigned long long>& hs = handles_[g];
  CUmemAccessDesc acc = {};
  acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  acc.location.id = device_;
  acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
  for (int l = 0; l < L_; ++l) {
    const CUdeviceptr at = (CUdeviceptr)(base_ + ((size_t)l * P_ + (size_t)g * G_) * bb_);
    CUmemGenericAllocationHandle h = 0;
    if (alloc_injected_failure() || v.create(&h, gbytes, &prop, 0) != CUDA_SUCCESS) {
      err = "KV pool: cuMemCreate failed (device memory)";
      unmap_group(g);
      return MAG_ERR_OOM;
    }
    if (v.map(at, gbytes, 0, h, 0) != CUDA_SUCCESS) {
      v.release(h);
      err = "KV pool: cuMemMap failed";
      unmap_group(g);
      return MAG_ERR_CUDA;
    }
    hs.push_back(h);
    if (v.access(at, gbytes, &acc, 1) != CUDA_SUCCESS) {
      err = "KV pool: cuMemSetAccess failed";
      unmap_group(g);
      return MAG_ERR_CUDA;
    }
  }
  for (int l = 0; l < L_; ++l) {
    const cudaError_t e = cudaMemsetAsync(base_ + ((size_t)l * P_ + (size_t)g * G_) * bb_, 0, gbytes, s);
    if (e != cudaSuccess) {
      err = std::string("KV pool: memset: ") + cudaGetErrorString(e);
      return MAG_ERR_CUDA;
    }
  }
  state_[g] = kMapped;
  used_[g] = 0;
  for (int64_t b = g * G_; b < (g + 1) * G_; ++b) free_set_.insert((int32_t)b);
  return MAG_OK;
}

// Unmaps whatever part of group g is mapped (handles_[g] holds the layers mapped so far, in order).
mag_status KvPool::unmap_group(int64_t g) {
  const Vmm& v = vmm();
  const size_t gbytes = (size_t)G_ * bb_;
  mag_status st = MAG_OK;
  std::vector<unsigned long long>& hs = handles_[g];
  for (size_t l = 0; l < hs.size(); ++l) {
    const CUdeviceptr at = (CUdeviceptr)(base_ + ((size_t)l * P_ + (size_t)g * G_) * bb_);
    if (v.unmap(at, gbytes) != CUDA_SUCCESS) st = MAG_ERR_CUDA;
    if (v.release(hs[l]) != CUDA_SUCCESS) st = MAG_ERR_CUDA;
  }
  hs.clear();
  if (state_[g] == kMapped)
    for (int64_t b = g * G_; b < (g + 1) * G_; ++b) free_set_.erase((int32_t)b);
  state_[g] = kUnmapped;
  if (st != MAG_OK) err = "KV pool: unmapping a group failed";
  return st;
}

void KvPool::revive(int64_t g) {
  state_[g] = kMapped;
  for (int64_t b = g * G_; b < (g + 1) * G_; ++b) free_set_.insert((int32_t)b);
}

int64_t KvPool::available() const {
  if (!elastic_) return (int64_t)fifo_.size();
  int64_t n = (int64_t)free_set_.size();
  for (int64_t g = 0; g < n_groups_; ++g)
    if (state_[g] != kMapped) n += G_;
  return n;
}

int64_t KvPool::mapped_blocks() const {
  if (!elastic_) return P_;
  int64_t n = 0;
  for (int64_t g = 0; g < n_groups_; ++g)
    if (state_[g] != kUnmapped) n += G_;
  return n;
}

bool KvPool::is_mapped(int32_t b) const {
  if (!elastic_) return b >= 0 && b < P_;
  return b >= 0 && b < P_ && state_[b / G_] == kMapped;
}

mag_status KvPool::reserve(int64_t n, cudaStream_t s) {
  if (n <= free_now()) return MAG_OK;
  if (n > available()) return MAG_ERR_KV_FULL;
  // the lowest groups not in use first: one on its way out comes back as it is, another is mapped
  for (int64_t g = 0; g < n_groups_ && free_now() < n; ++g) {
    if (state_[g] == kReleasing) revive(g);
    if (state_[g] == kUnmapped) {
      const mag_status st = map_group(g, s);
      if (st != MAG_OK) return st;
    }
  }
  return MAG_OK;
}

int32_t KvPool::pop() {
  if (!elastic_) {
    const int32_t b = fifo_.front();
    fifo_.pop_front();
    return b;
  }
  const int32_t b = *free_set_.begin();
  free_set_.erase(free_set_.begin());
  ++used_[b / G_];
  return b;
}

void KvPool::push(int32_t b) {
  if (!elastic_) {
    fifo_.push_back(b);
    return;
  }
  --used_[b / G_];
  free_set_.insert(b);
}

mag_status KvPool::set_hot(int64_t blocks, cudaStream_t s, const std::function<bool(int64_t)>& referenced) {
  if (!elastic_) return MAG_OK;
  hot_groups_ = std::min<int64_t>(std::max<int64_t>((blocks + G_ - 1) / G_, 1), n_groups_);
  for (int64_t g = 0; g < hot_groups_; ++g) {
    if (state_[g] == kReleasing) revive(g);
    if (state_[g] == kUnmapped) {
      const mag_status st = map_group(g, s);
      if (st != MAG_OK) return st;
    }
  }
  return trim(s, referenced);
}

mag_status KvPool::trim(cudaStream_t s, const std::function<bool(int64_t)>& referenced) {
  if (!elastic_) return MAG_OK;
  for (int64_t g = 0; g < n_groups_; ++g) {
    if (state_[g] != kReleasing) continue;
    const cudaError_t q = cudaEventQuery(release_ev_[g]);
    if (q == cudaErrorNotReady) continue;
    if (q != cudaSuccess) {
      err = std::string("KV pool: release event: ") + cudaGetErrorString(q);
      return MAG_ERR_CUDA;
    }
    const mag_status st = unmap_group(g);
    if (st != MAG_OK) return st;
  }
  for (int64_t g = hot_groups_; g < n_groups_; ++g) {
    if (state_[g] != kMapped || used_[g] != 0) continue;
    if (referenced && referenced(g)) {
      err = "KV pool: a group with no blocks in use is still listed by a session";
      return MAG_ERR_CUDA;
    }
    if (!release_ev_[g] && cudaEventCreateWithFlags(&release_ev_[g], cudaEventDisableTiming) != cudaSuccess) {
      err = "KV pool: event create failed";
      return MAG_ERR_CUDA;
    }
    const cudaError_t e = cudaEventRecord(release_ev_[g], s);
    if (e != cudaSuccess) {
      err = std::string("KV pool: event record: ") + cudaGetErrorString(e);
      return MAG_ERR_CUDA;
    }
    for (int64_t b = g * G_; b < (g + 1) * G_; ++b) free_set_.erase((int32_t)b);
    state_[g] = kReleasing;
  }
  return MAG_OK;
}

}  // namespace mag
