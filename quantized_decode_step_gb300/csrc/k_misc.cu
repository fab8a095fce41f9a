// Load-time W4 quantiser, step prologue and the no-LM-head output.
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

// Step prologue: write this step's block-table entries and load the fp16
// hidden inputs into the fp32 residual stream.
__global__ void step_begin_kernel(const StepArgs* __restrict__ st, float* __restrict__ r, int D,
                                  int32_t* __restrict__ tables, int table_stride) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  if (b == 0 && threadIdx.x < st->n_upd)
    tables[(int64_t)st->upd_sess[threadIdx.x] * table_stride + st->upd_idx[threadIdx.x]] = st->upd_blk[threadIdx.x];
  for (int i = threadIdx.x; i < D; i += blockDim.x)
    r[(int64_t)b * D + i] = __half2float(st->hidden_in[(int64_t)b * D + i]);
}

// No LM head: the output is the fp16 hidden state.
__global__ void final_hidden_kernel(const StepArgs* __restrict__ st, const float* __restrict__ r, int D) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  __half* out = reinterpret_cast<__half*>(st->out);
  for (int i = threadIdx.x; i < D; i += blockDim.x) out[(int64_t)b * D + i] = __float2half_rn(r[(int64_t)b * D + i]);
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
                              int table_stride, int batch) {
  return launch_plain(L, step_begin_kernel, dim3(batch), dim3(256), step, r, D, tables, table_stride);
}

cudaError_t launch_final_hidden(const Launch& L, const StepArgs* step, const float* r, int D, int batch) {
  return launch_plain(L, final_hidden_kernel, dim3(batch), dim3(256), step, r, D);
}

}  // namespace mag
