// Load-time W4 quantiser and the decode-step prologue.
#include "kernels.h"

namespace mag {

namespace {

// One thread per 32-value group ("5. Core modules" 5.1, 4-bit weights):
// m = fp16(min), s = fp16((max - min) / 15) with an fp32 subtract and IEEE
// divide, code = clamp(rint((x - m) / s), 0, 15) in fp32 (0 when s == 0);
// byte j holds codes 2j (low nibble) and 2j+1 (high nibble); a ragged last
// group covers the remaining values and pads with code 0. Min and max are
// taken in index order, so the bytes are fixed by the rule alone.
__global__ void quantize_w4g32_kernel(const float* __restrict__ src, int64_t rows, int64_t cols, int64_t groups,
                                      uint8_t* __restrict__ codes, __half2* __restrict__ sm) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= rows * groups) return;
  const int64_t r = gid / groups, g = gid - r * groups;
  const float* x = src + r * cols + g * 32;
  const int n = (int)min((int64_t)32, cols - g * 32);
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = i < n ? x[i] : 0.f;
  float lo = v[0], hi = v[0];
  for (int i = 1; i < n; ++i) {
    if (v[i] < lo) lo = v[i];
    if (v[i] > hi) hi = v[i];
  }
  __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.0f));
  __half m16 = __float2half_rn(lo);
  float s = __half2float(s16), m = __half2float(m16);
  uint32_t words[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    int q = 0;
    if (i < n && s != 0.0f) {
      q = (int)rintf(__fdiv_rn(__fsub_rn(v[i], m), s));
      q = max(0, min(15, q));
    }
    words[i >> 3] |= (uint32_t)q << (4 * (i & 7));
  }
  *reinterpret_cast<uint4*>(codes + (r * groups + g) * 16) = make_uint4(words[0], words[1], words[2], words[3]);
  sm[r * groups + g] = __halves2half2(s16, m16);
}

// Step prologue (one block per token): write this step's block-table entries,
// load the fp16 hidden input into the fp32 residual stream and store its sum
// of squares in ss_part[0][b] for the first layer's RMSNorm.
__global__ void step_begin_kernel(const StepArgs* __restrict__ st, float* __restrict__ r, int D,
                                  int32_t* __restrict__ tables, int table_stride, float* __restrict__ ss_part) {
  __shared__ float s_red[32];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (b == 0 && tid < st->n_upd)
    tables[(int64_t)st->upd_sess[tid] * table_stride + st->upd_idx[tid]] = st->upd_blk[tid];
  const __half* hin = st->hidden_in + (int64_t)b * D;
  float ss = 0.f;
  for (int u = tid; u < D / 8; u += blockDim.x) {
    const uint4 v = *reinterpret_cast<const uint4*>(hin + 8 * u);
    const __half* h = reinterpret_cast<const __half*>(&v);
    float f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      f[e] = __half2float(h[e]);
      ss += f[e] * f[e];
    }
    *reinterpret_cast<float4*>(r + (int64_t)b * D + 8 * u) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(r + (int64_t)b * D + 8 * u + 4) = make_float4(f[4], f[5], f[6], f[7]);
  }
  ss = warp_sum(ss);
  if (lane == 0) s_red[warp] = ss;
  __syncthreads();
  if (tid == 0) {
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_red[w];
    ss_part[b] = tot;  // entry 0 of token b (row stride MAG_MAX_BATCH)
  }
}

// Debug canaries: every 32-bit word of every arena tensor's two bands must still hold the pattern; a changed
// band sets kErrCanary and the tensor's bit in the error word.
__global__ void arena_check_kernel(const ArenaCheck a) {
  pdl_wait();
  pdl_trigger();
  constexpr int W = kCanaryBand / 4;  // words per band
  const uint32_t pattern = (uint32_t)kCanaryByte * 0x01010101u;
  for (int i = threadIdx.x; i < a.n * 2 * W; i += blockDim.x) {
    const int tsr = i / (2 * W), r = i - tsr * 2 * W, side = r / W, w = r - side * W;
    const uint32_t v = __ldcg(reinterpret_cast<const unsigned int*>(a.base + a.band[tsr][side]) + w);
    if (v != pattern) atomicOr(a.err, kErrCanary | (1u << (kErrCanaryShift + tsr)));
  }
}

// No LM head: the output is the fp16 hidden state.
__global__ void final_hidden_kernel(const StepArgs* __restrict__ st, const float* __restrict__ r, int D) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  __half* out = reinterpret_cast<__half*>(st->out);
  for (int i = threadIdx.x; i < D; i += blockDim.x) out[(int64_t)b * D + i] = __float2half_rn(r[(int64_t)b * D + i]);
}

// Row pair (r_g, r_g8) of slot g of tile mt under a tile map.
__device__ __forceinline__ void tile_rows(int map, int map_arg, int mt, int g, int& rg, int& rg8) {
  if (map == MAP_SWIGLU) {
    rg = mt * 8 + g;
    rg8 = map_arg + mt * 8 + g;
  } else if (map == MAP_QKV) {
    const int tph = map_arg / 16, head = mt / tph;
    rg = head * map_arg + 8 * (mt - head * tph) + g;
    rg8 = rg + map_arg / 2;
  } else {
    rg = mt * 16 + g;
    rg8 = rg + 8;
  }
}

// One thread per (tile, chunk, lane): the lane's 16 bytes of codes, and for
// t == 0 the 16 bytes of (scale, min) of its row pair. dir 0: canonical ->
// tiles, 1: tiles -> canonical.
__global__ void w4_tiles_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int N, int K, int map,
                                int map_arg, int dir) {
  const int G = (K + 31) / 32, C = (K + 63) / 64, n_mt = N / 16;
  const int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (id >= (int64_t)n_mt * C * 32) return;
  const int lane = (int)(id & 31), g = lane >> 2, t = lane & 3;
  const int64_t tc = id >> 5;
  const int mt = (int)(tc / C), c = (int)(tc - (int64_t)mt * C);
  int rg, rg8;
  tile_rows(map, map_arg, mt, g, rg, rg8);
  const int64_t code_bytes = (int64_t)N * G * 16;
  uint8_t* tile = (dir == 0 ? dst : const_cast<uint8_t*>(src)) + tc * kTileBytes;
  const int rows[2] = {rg, rg8};
  for (int h = 0; h < 2; ++h)
    for (int q = 0; q < 2; ++q) {
      const int grp = 2 * c + q;
      uint32_t* tw = reinterpret_cast<uint32_t*>(tile + lane * 16) + 2 * h + q;
      if (dir == 0) {
        *tw = grp < G ? *reinterpret_cast<const uint32_t*>(src + (int64_t)rows[h] * G * 16 + grp * 16 + 4 * t) : 0u;
      } else if (grp < G) {
        *reinterpret_cast<uint32_t*>(dst + (int64_t)rows[h] * G * 16 + grp * 16 + 4 * t) = *tw;
      }
    }
  if (t == 0) {
    for (int h = 0; h < 2; ++h)
      for (int q = 0; q < 2; ++q) {
        const int grp = 2 * c + q;
        uint32_t* ts = reinterpret_cast<uint32_t*>(tile + 512 + g * 16) + 2 * h + q;
        const int64_t ci = code_bytes + ((int64_t)rows[h] * G + grp) * 4;
        if (dir == 0) {
          *ts = grp < G ? *reinterpret_cast<const uint32_t*>(src + ci) : 0u;
        } else if (grp < G) {
          *reinterpret_cast<uint32_t*>(dst + ci) = *ts;
        }
      }
  }
}


// One thread per (tile, chunk, lane, row half): 16 fp16 values of row g (or g+8).
__global__ void f16_tiles_kernel(const __half* __restrict__ src, int N, int K, uint8_t* __restrict__ dst) {
  const int C = (K + 63) / 64, n_mt = N / 16;
  const int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (id >= (int64_t)n_mt * C * 64) return;
  const int h = (int)(id & 1), lane = (int)((id >> 1) & 31), g = lane >> 2, t = lane & 3;
  const int64_t tc = id >> 6;
  const int mt = (int)(tc / C), c = (int)(tc - (int64_t)mt * C);
  const int64_t row = (int64_t)mt * 16 + g + 8 * h;
  const int k0 = c * 64 + t * 16;
  __half v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = k0 + j < K ? src[row * K + k0 + j] : __float2half_rn(0.f);
  uint4* o = reinterpret_cast<uint4*>(dst + tc * 2048 + lane * 64 + h * 32);
  o[0] = *reinterpret_cast<uint4*>(v);
  o[1] = *reinterpret_cast<uint4*>(v + 8);
}

template <typename K, typename... Args>
cudaError_t launch_plain(const Launch& L, K kern, dim3 grid, dim3 block, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.counter) ++*L.counter;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

cudaError_t launch_quantize_w4g32(cudaStream_t s, const float* src, int64_t rows, int64_t cols, uint8_t* codes,
                                  __half2* sm) {
  const int64_t groups = (cols + 31) / 32;
  const int64_t n = rows * groups;
  if (n == 0) return cudaSuccess;
  const int threads = 128;
  quantize_w4g32_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(src, rows, cols, groups, codes,
                                                                                      sm);
  return cudaGetLastError();
}

cudaError_t launch_step_begin(const Launch& L, const StepArgs* step, float* r, int D, int32_t* tables,
                              int table_stride, int batch, float* ss_part) {
  return launch_plain(L, step_begin_kernel, dim3(batch), dim3(256), step, r, D, tables, table_stride, ss_part);
}

cudaError_t launch_arena_check(const Launch& L, const ArenaCheck& a) {
  if (a.n < 1 || a.n > 16) return cudaErrorInvalidValue;
  return launch_plain(L, arena_check_kernel, dim3(1), dim3(256), a);
}

cudaError_t launch_final_hidden(const Launch& L, const StepArgs* step, const float* r, int D, int batch) {
  return launch_plain(L, final_hidden_kernel, dim3(batch), dim3(256), step, r, D);
}

static cudaError_t launch_tiles(cudaStream_t s, const uint8_t* src, uint8_t* dst, int N, int K, int map, int map_arg,
                                int dir) {
  const int64_t n = (int64_t)(N / 16) * ((K + 63) / 64) * 32;
  if (n == 0) return cudaSuccess;
  w4_tiles_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(src, dst, N, K, map, map_arg, dir);
  return cudaGetLastError();
}

cudaError_t launch_w4_to_tiles(cudaStream_t s, const uint8_t* canon, int N, int K, int map, int map_arg,
                               uint8_t* tiles) {
  return launch_tiles(s, canon, tiles, N, K, map, map_arg, 0);
}

cudaError_t launch_w4_from_tiles(cudaStream_t s, const uint8_t* tiles, int N, int K, int map, int map_arg,
                                 uint8_t* canon) {
  return launch_tiles(s, tiles, canon, N, K, map, map_arg, 1);
}

}  // namespace mag

namespace mag {

cudaError_t launch_f16_to_tiles(cudaStream_t s, const __half* src, int N, int K, uint8_t* tiles) {
  const int64_t n = (int64_t)(N / 16) * ((K + 63) / 64) * 64;
  if (n == 0) return cudaSuccess;
  f16_tiles_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(src, N, K, tiles);
  return cudaGetLastError();
}
}  // namespace mag
