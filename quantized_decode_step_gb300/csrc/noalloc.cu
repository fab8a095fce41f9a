// Loading an fp32 projection without allocating device memory.
//
// The ordinary fp32 load quantises the whole projection into a stream-ordered
// scratch copy in W4G32 bytes (cudaMallocAsync of up to N*K*5/8 bytes, 73 MB
// for an 8B gate-up) and then tiles it. A caller that sized the KV pool to
// fill the HBM left after the weights, or that forbids device allocation
// after start-up, cannot make that allocation. This path instead walks the
// projection in slabs of whole tiles through one fixed scratch buffer that is
// part of the library image: quantise the slab's rows into the scratch, tile
// them into place, next slab. The kernels are the ordinary load's, unchanged;
// each slab is a self-contained smaller projection of the same tile map.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "kernels.h"
#include "noalloc.h"

// Scratch of the no-alloc fp32 load: one per device, shared by every context.
static __device__ __align__(256) uint8_t mag_noalloc_scratch[mag::kNoAllocScratchBytes];

namespace mag {

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
struct DeviceScratch {
  unsigned long long ctx_id = 0;  // driver id of the context the address belongs to
  uint8_t* ptr = nullptr;
};
DeviceScratch g_scratch[kMaxDevices];

// Driver id of the calling thread's current context (unique for the process's lifetime, so a primary
// context created again after a device reset gets a new one); 0 when none is current or the driver
// calls are unavailable.
unsigned long long current_ctx_id() {
  static decltype(&::cuCtxGetCurrent) get_current = nullptr;
  static decltype(&::cuCtxGetId) get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", reinterpret_cast<void**>(&get_current), 12000,
                                         cudaEnableDefault, &q) != cudaSuccess || q != cudaDriverEntryPointSuccess)
      get_current = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", reinterpret_cast<void**>(&get_id), 12000, cudaEnableDefault,
                                         &q) != cudaSuccess || q != cudaDriverEntryPointSuccess)
      get_id = nullptr;
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch on the current device: looked up (cudaGetSymbolAddress, with the device
// current) the first time a device's context is seen, and again if that context was replaced since (a
// device reset reloads the library's module, possibly elsewhere). A cached address is only reused for the
// context it was looked up in.
cudaError_t scratch_on_current_device(uint8_t** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceScratch& d = g_scratch[dev];
  const unsigned long long id = current_ctx_id();
  if (!d.ptr || id == 0 || id != d.ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, mag_noalloc_scratch);
    if (e != cudaSuccess) return e;
    d.ptr = static_cast<uint8_t*>(p);
    d.ctx_id = current_ctx_id();  // the lookup made the device's primary context current if none was
  }
  *out = d.ptr;
  return cudaSuccess;
}

}  // namespace

int noalloc_slab_tiles(int K, int map, int map_arg) {
  const int64_t G = (K + 31) / 32;
  const int64_t per_tile = 16 * G * 20;  // 16 rows x (16 B of codes + 4 B of (scale, min)) per group
  const int64_t unit = map == MAP_QKV ? map_arg / 16 : 1;  // QKV slabs hold whole heads
  int64_t n = (int64_t)kNoAllocScratchBytes / per_tile;
  n -= n % unit;
  return n < unit ? 0 : (int)std::min<int64_t>(n, 1 << 30);
}

cudaError_t load_f32_noalloc(cudaStream_t s, const float* src, int N, int K, int map, int map_arg, uint8_t* tiles) {
  const int slab = noalloc_slab_tiles(K, map, map_arg);
  if (slab == 0) return cudaErrorInvalidValue;
  uint8_t* scratch = nullptr;
  cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) return e;
  const int64_t G = (K + 31) / 32, C = (K + 63) / 64, n_mt = N / 16;
  for (int64_t mt0 = 0; mt0 < n_mt; mt0 += slab) {
    const int n = (int)std::min<int64_t>(slab, n_mt - mt0);
    const int64_t rows = 16 * (int64_t)n;  // rows of the slab's sub-projection
    uint8_t* codes = scratch;
    uint8_t* sm = scratch + rows * G * 16;
    int sub_arg = map_arg;
    if (map == MAP_SWIGLU) {
      // tiles [mt0, mt0 + n) pair gate rows 8 mt0 + i with up rows F + 8 mt0 + i:
      // the sub-projection is [those 8n gate rows; those 8n up rows], its F = 8n
      const int64_t h = 8 * (int64_t)n;
      e = launch_quantize_w4g32(s, src + 8 * mt0 * (int64_t)K, h, K, codes, reinterpret_cast<__half2*>(sm));
      if (e == cudaSuccess)
        e = launch_quantize_w4g32(s, src + ((int64_t)map_arg + 8 * mt0) * K, h, K, codes + h * G * 16,
                                  reinterpret_cast<__half2*>(sm + h * G * 4));
      sub_arg = (int)h;
    } else {
      // plain rows, or (QKV) whole heads: rows 16 mt0 .. 16 (mt0 + n)
      e = launch_quantize_w4g32(s, src + 16 * mt0 * (int64_t)K, rows, K, codes, reinterpret_cast<__half2*>(sm));
    }
    if (e == cudaSuccess) e = launch_w4_to_tiles(s, scratch, (int)rows, K, map, sub_arg, tiles + mt0 * C * kTileBytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace mag
