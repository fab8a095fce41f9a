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
// load the fp16 hidden input into the fp32 residual stream, and RMSNorm it for
// the first layer's QKV projection ("5. Core modules" 5.1, pre-norm): xn in
// the W4 activation unit order (x0,x4,x1,x5,x2,x6,x3,x7) plus its 32-value
// group sums.
__global__ void step_begin_kernel(const StepArgs* __restrict__ st, float* __restrict__ r, int D,
                                  int32_t* __restrict__ tables, int table_stride, const __half* __restrict__ gamma,
                                  float eps, __half* __restrict__ xn, float* __restrict__ xn_sum) {
  __shared__ float s_red[32];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (b == 0 && tid < st->n_upd)
    tables[(int64_t)st->upd_sess[tid] * table_stride + st->upd_idx[tid]] = st->upd_blk[tid];
  const __half* hin = st->hidden_in + (int64_t)b * D;
  const int units = D / 8;
  float ss = 0.f;
  for (int u = tid; u < units; u += blockDim.x) {
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
    s_red[0] = 1.0f / sqrtf(tot / (float)D + eps);
  }
  __syncthreads();
  const float inv = s_red[0];
  for (int base = 0; base < units; base += blockDim.x) {  // warp-uniform trips: quads share a group
    const int u = base + tid;
    float s = 0.f;
    if (u < units) {
      const uint4 v = *reinterpret_cast<const uint4*>(hin + 8 * u);
      const uint4 gg = *reinterpret_cast<const uint4*>(gamma + 8 * u);
      const __half* h = reinterpret_cast<const __half*>(&v);
      const __half* gh = reinterpret_cast<const __half*>(&gg);
      __half o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const __half x = __float2half_rn(__half2float(h[e]) * inv * __half2float(gh[e]));
        o[e < 4 ? 2 * e : 2 * (e - 4) + 1] = x;
        s += __half2float(x);
      }
      *reinterpret_cast<uint4*>(xn + (int64_t)b * D + 8 * u) = *reinterpret_cast<uint4*>(o);
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    if (u < units && (u & 3) == 0) xn_sum[(int64_t)b * (D / 32) + u / 4] = s;
  }
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
                              int table_stride, int batch, const __half* gamma, float eps, __half* xn,
                              float* xn_sum) {
  return launch_plain(L, step_begin_kernel, dim3(batch), dim3(256), step, r, D, tables, table_stride, gamma, eps,
                      xn, xn_sum);
}

}  // namespace mag
