// The fp32 projection load that allocates nothing (noalloc.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mag {

// Size of the per-device scratch the no-alloc load walks a projection through.
constexpr size_t kNoAllocScratchBytes = 4u << 20;

// Tiles per slab for a projection of reduction length K under a tile map, or 0
// when one slab (one tile, or one head of tiles for QKV) does not fit the scratch.
int noalloc_slab_tiles(int K, int map, int map_arg);

// Quantise fp32 [N][K] and write its tiles, slab by slab through the scratch,
// on stream s. Calls that overlap in time on one device race on the scratch.
cudaError_t load_f32_noalloc(cudaStream_t s, const float* src, int N, int K, int map, int map_arg, uint8_t* tiles);

}  // namespace mag
