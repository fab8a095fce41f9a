// W4A16 (and fp16) matrix-vector products of the decode step on mma.sync.
//
// y[b][n] = sum_k deq(W)[n][k] * x[b][k] for a handful of tokens b, with the
// weights streamed once from HBM in the packed 4-bit group-32 layout the
// library takes at load time ("5. Core modules" 5.1: 4-bit weights with FP16
// activations). No repacking: each lane reads 8 bytes of two rows per 64-wide
// k-chunk, turns the nibbles into fp16 with a LOP3 into the mantissa of 1024
// (the int4-to-fp16 conversion of Kim et al., "Who Says Elephants Can't Run",
// 2022), applies scale and min with one HFMA2 and feeds m16n8k16 tensor-core
// MMAs with fp32 accumulators. The activations sit in shared memory in the
// k order those fragments imply, so one 128-bit shared load gives a lane the
// B fragments of two k-steps.
//
// Fused around the product:
//   prologue  RMSNorm of the fp32 residual ("5. Core modules" 5.1, pre-norm);
//   epilogue  fp16 store / fp32 residual add / SwiGLU of interleaved gate-up.
// Weight loads for the first chunks are issued before the programmatic-
// dependent-launch wait, so they overlap the previous kernel's tail.
#include "kernels.h"

namespace mag {

namespace {

constexpr int kStages = 4;

struct W4Stage {
  uint2 wg, wg8;
  uint32_t sg, sg8;
};
struct F16Stage {
  uint4 g0, g1, h0, h1;
};

template <int WFMT>
struct StageT;
template <>
struct StageT<W_W4> {
  using type = W4Stage;
};
template <>
struct StageT<W_F16> {
  using type = F16Stage;
};

__device__ __forceinline__ void load_stage(W4Stage& st, const GemvArgs& a, int row_g, int row_g8, int c, int t) {
  int grp = 2 * c + (t >> 1);
  if (grp < a.sm_row) {
    const uint8_t* pg = a.w + (int64_t)row_g * a.w_row_bytes + c * 32 + t * 8;
    const uint8_t* pg8 = a.w + (int64_t)row_g8 * a.w_row_bytes + c * 32 + t * 8;
    st.wg = ldg_stream_u2(pg);
    st.wg8 = ldg_stream_u2(pg8);
    st.sg = ldg_nc_u32(a.sm + (int64_t)row_g * a.sm_row + grp);
    st.sg8 = ldg_nc_u32(a.sm + (int64_t)row_g8 * a.sm_row + grp);
  } else {
    st.wg = make_uint2(0, 0);
    st.wg8 = make_uint2(0, 0);
    st.sg = 0;
    st.sg8 = 0;
  }
}

__device__ __forceinline__ void load_stage(F16Stage& st, const GemvArgs& a, int row_g, int row_g8, int c, int t) {
  int k = c * 64 + t * 16;
  if (k < a.K) {
    const uint8_t* pg = a.w + (int64_t)row_g * a.w_row_bytes + (int64_t)k * 2;
    const uint8_t* pg8 = a.w + (int64_t)row_g8 * a.w_row_bytes + (int64_t)k * 2;
    st.g0 = ldg_stream_u4(pg);
    st.g1 = ldg_stream_u4(pg + 16);
    st.h0 = ldg_stream_u4(pg8);
    st.h1 = ldg_stream_u4(pg8 + 16);
  } else {
    st.g0 = st.g1 = st.h0 = st.h1 = make_uint4(0, 0, 0, 0);
  }
}

// Nibble pairs of one 32-bit word of codes (canonical order: k0 in bits 0-3,
// k1 in bits 4-7, ..., k7 in bits 28-31) as fp16 pairs times scale plus min:
//   E0 = (k0, k4), E1 = (k1, k5), E2 = (k2, k6), E3 = (k3, k7).
struct Deq4 {
  uint32_t e0, e1, e2, e3;
};
__device__ __forceinline__ Deq4 dequant_word(uint32_t w, __half2 s2, __half2 m2) {
  const __half2 k1024 = __float2half2_rn(1024.0f);
  const __half2 k1_16 = __float2half2_rn(0.0625f);
  const __half2 km64 = __float2half2_rn(-64.0f);
  uint32_t w2 = w >> 8;
  __half2 q0 = __hsub2(u32_as_h2(lop3_and_or(w, 0x000F000Fu, 0x64006400u)), k1024);
  __half2 q1 = __hfma2(u32_as_h2(lop3_and_or(w, 0x00F000F0u, 0x64006400u)), k1_16, km64);
  __half2 q2 = __hsub2(u32_as_h2(lop3_and_or(w2, 0x000F000Fu, 0x64006400u)), k1024);
  __half2 q3 = __hfma2(u32_as_h2(lop3_and_or(w2, 0x00F000F0u, 0x64006400u)), k1_16, km64);
  Deq4 d;
  d.e0 = h2_as_u32(__hfma2(q0, s2, m2));
  d.e1 = h2_as_u32(__hfma2(q1, s2, m2));
  d.e2 = h2_as_u32(__hfma2(q2, s2, m2));
  d.e3 = h2_as_u32(__hfma2(q3, s2, m2));
  return d;
}

template <int NT>
__device__ __forceinline__ void compute_stage(const W4Stage& st, float (&acc)[2][4], const uint4 (&xb)[2][2]) {
  __half2 sgm = u32_as_h2(st.sg), sg8m = u32_as_h2(st.sg8);
  __half2 s_g = __low2half2(sgm), m_g = __high2half2(sgm);
  __half2 s_g8 = __low2half2(sg8m), m_g8 = __high2half2(sg8m);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t w = q ? st.wg.y : st.wg.x;
    uint32_t v = q ? st.wg8.y : st.wg8.x;
    Deq4 dg = dequant_word(w, s_g, m_g);
    Deq4 dv = dequant_word(v, s_g8, m_g8);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      // k-step 2q: a0 = E0(row g), a1 = E0(row g+8), a2 = E1(row g), a3 = E1(row g+8)
      mma_16816(acc[nt], dg.e0, dv.e0, dg.e1, dv.e1, xb[nt][q].x, xb[nt][q].y);
      // k-step 2q+1: E2 / E3
      mma_16816(acc[nt], dg.e2, dv.e2, dg.e3, dv.e3, xb[nt][q].z, xb[nt][q].w);
    }
  }
}

template <int NT>
__device__ __forceinline__ void compute_stage(const F16Stage& st, float (&acc)[2][4], const uint4 (&xb)[2][2]) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    mma_16816(acc[nt], st.g0.x, st.h0.x, st.g0.y, st.h0.y, xb[nt][0].x, xb[nt][0].y);
    mma_16816(acc[nt], st.g0.z, st.h0.z, st.g0.w, st.h0.w, xb[nt][0].z, xb[nt][0].w);
    mma_16816(acc[nt], st.g1.x, st.h1.x, st.g1.y, st.h1.y, xb[nt][1].x, xb[nt][1].y);
    mma_16816(acc[nt], st.g1.z, st.h1.z, st.g1.w, st.h1.w, xb[nt][1].z, xb[nt][1].w);
  }
}

// 8 consecutive fp16 activations -> shared-memory order of the W4 fragments
// (k0,k4,k1,k5,k2,k6,k3,k7) or natural order for fp16 weights.
template <int WFMT>
__device__ __forceinline__ uint4 permute8(uint4 v) {
  if (WFMT == W_F16) return v;
  uint4 o;
  o.x = __byte_perm(v.x, v.z, 0x5410);  // (k0, k4)
  o.y = __byte_perm(v.x, v.z, 0x7632);  // (k1, k5)
  o.z = __byte_perm(v.y, v.w, 0x5410);  // (k2, k6)
  o.w = __byte_perm(v.y, v.w, 0x7632);  // (k3, k7)
  return o;
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 o;
  o.x = h2_as_u32(__floats2half2_rn(f[0], f[1]));
  o.y = h2_as_u32(__floats2half2_rn(f[2], f[3]));
  o.z = h2_as_u32(__floats2half2_rn(f[4], f[5]));
  o.w = h2_as_u32(__floats2half2_rn(f[6], f[7]));
  return o;
}

template <int NT, int WFMT, int XMODE, int EPI>
__global__ void __launch_bounds__(256) gemv_kernel(const GemvArgs a) {
  using Stage = typename StageT<WFMT>::type;
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int mt_local = warp % a.mpc, kw = warp / a.mpc;
  const int mt = blockIdx.x * a.mpc + mt_local;
  const bool mt_ok = mt < a.n_mtiles;
  const int c_begin = blockIdx.y * a.chunks_per_cta;
  const int c_end = min(c_begin + a.chunks_per_cta, a.n_chunks);
  const int n_cc = c_end - c_begin;  // chunks of this block
  const int B = a.batch;

  int row_g, row_g8;
  if (EPI == EPI_SWIGLU) {
    row_g = mt * 8 + g;
    row_g8 = a.swiglu_f + mt * 8 + g;
  } else {
    row_g = mt * 16 + g;
    row_g8 = row_g + 8;
  }

  // this warp's chunks: c_begin + kw + i * wk
  const int n_my = (mt_ok && kw < n_cc) ? (n_cc - kw + a.wk - 1) / a.wk : 0;
  Stage st[kStages];
#pragma unroll
  for (int u = 0; u < kStages; ++u)
    if (u < n_my) load_stage(st[u], a, row_g, row_g8, c_begin + kw + u * a.wk, t);

  pdl_wait();
  pdl_trigger();

  // ---- stage the activations of this block's k-range
  const int xrow = n_cc * 64 + 8;  // halves per token row (+16 B against bank conflicts)
  __half* xs = reinterpret_cast<__half*>(smem);
  float* misc = reinterpret_cast<float*>(smem + (size_t)B * xrow * 2);
  const int k0 = c_begin * 64;
  if (XMODE == X_NORM) {
    // RMSNorm: inv[b] = 1 / sqrt(mean(r^2) + eps) over the full row
    float ss[MAG_MAX_BATCH];
    for (int b = 0; b < B; ++b) ss[b] = 0.f;
    for (int k = tid * 4; k < a.K; k += blockDim.x * 4) {
      for (int b = 0; b < B; ++b) {
        float4 v = *reinterpret_cast<const float4*>(a.r + (int64_t)b * a.ldr + k);
        ss[b] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
    }
    for (int b = 0; b < B; ++b) {
      float v = warp_sum(ss[b]);
      if (lane == 0) misc[warp * MAG_MAX_BATCH + b] = v;
    }
    __syncthreads();
    if (tid < B) {
      float tot = 0.f;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += misc[w * MAG_MAX_BATCH + tid];
      misc[8 * MAG_MAX_BATCH + tid] = 1.0f / sqrtf(tot / (float)a.K + a.eps);
    }
    __syncthreads();
  }
  const int units = n_cc * 8;  // 8-wide units of the k-range
  for (int idx = tid; idx < units * B; idx += blockDim.x) {
    int b = idx / units, u = idx - b * units;
    int k = k0 + u * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (k < a.K) {
      if (XMODE == X_F16) {
        v = *reinterpret_cast<const uint4*>(a.x + (int64_t)b * a.ldx + k);
      } else {
        float inv = misc[8 * MAG_MAX_BATCH + b];
        float4 r0 = *reinterpret_cast<const float4*>(a.r + (int64_t)b * a.ldr + k);
        float4 r1 = *reinterpret_cast<const float4*>(a.r + (int64_t)b * a.ldr + k + 4);
        uint4 gg = *reinterpret_cast<const uint4*>(a.gamma + k);
        const __half* gh = reinterpret_cast<const __half*>(&gg);
        float f[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        for (int i = 0; i < 8; ++i) f[i] = f[i] * inv * __half2float(gh[i]);
        v = pack8(f);
      }
    }
    *reinterpret_cast<uint4*>(xs + (size_t)b * xrow + u * 8) = permute8<WFMT>(v);
  }
  __syncthreads();

  // ---- main loop
  float acc[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;

  for (int i = 0; i < n_my; i += kStages) {
#pragma unroll
    for (int u = 0; u < kStages; ++u) {
      if (i + u < n_my) {
        Stage cur = st[u];
        int c = c_begin + kw + (i + u) * a.wk;
        if (i + u + kStages < n_my) load_stage(st[u], a, row_g, row_g8, c + kStages * a.wk, t);
        uint4 xb[2][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          int tok = g + nt * 8;
          if (tok < B) {
            const uint4* p = reinterpret_cast<const uint4*>(xs + (size_t)tok * xrow + (c - c_begin) * 64 + t * 16);
            xb[nt][0] = p[0];
            xb[nt][1] = p[1];
          } else {
            xb[nt][0] = xb[nt][1] = make_uint4(0, 0, 0, 0);
          }
        }
        compute_stage<NT>(cur, acc, xb);
      }
    }
  }

  // ---- reduce the wk warps of each m-tile
  if (a.wk > 1) {
    __syncthreads();  // xs no longer needed: reuse it
    float* red = reinterpret_cast<float*>(smem);
    if (kw > 0) {
      float* p = red + (((size_t)(kw - 1) * a.mpc + mt_local) * 32 + lane) * 8;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) p[nt * 4 + i] = acc[nt][i];
    }
    __syncthreads();
    if (kw == 0) {
      for (int w = 1; w < a.wk; ++w) {
        const float* p = red + (((size_t)(w - 1) * a.mpc + mt_local) * 32 + lane) * 8;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[nt][i] += p[nt * 4 + i];
      }
    }
  }

  // ---- reduce across k-split blocks: the last block to arrive sums in split order
  if (a.ks > 1) {
    if (kw == 0 && mt_ok) {
      float* p = a.partial + (((size_t)blockIdx.y * a.n_mtiles + mt) * 32 + lane) * (4 * NT);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float4*>(p + nt * 4) = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
    }
    __threadfence();
    __syncthreads();
    __shared__ int s_last;
    if (tid == 0) {
      unsigned prev = atomicAdd(a.counters + blockIdx.x, 1u);
      s_last = (prev == (unsigned)(a.ks - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (kw == 0 && mt_ok) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
      for (int s = 0; s < a.ks; ++s) {
        const float* p = a.partial + (((size_t)s * a.n_mtiles + mt) * 32 + lane) * (4 * NT);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float4 v = __ldcg(reinterpret_cast<const float4*>(p + nt * 4));
          acc[nt][0] += v.x;
          acc[nt][1] += v.y;
          acc[nt][2] += v.z;
          acc[nt][3] += v.w;
        }
      }
    }
    if (tid == 0) a.counters[blockIdx.x] = 0;
  }

  // ---- epilogue
  if (kw != 0 || !mt_ok) return;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      int tok = nt * 8 + 2 * t + j;
      if (tok >= B) continue;
      float lo = acc[nt][j], hi = acc[nt][j + 2];  // rows g and g + 8
      if (EPI == EPI_SWIGLU) {
        int col = mt * 8 + g;
        float act = lo / (1.0f + expf(-lo)) * hi;
        a.out_h[(int64_t)tok * a.ldo + col] = __float2half_rn(act);
      } else if (EPI == EPI_RESID) {
        float* o = a.out_r + (int64_t)tok * a.ldo + mt * 16 + g;
        o[0] += lo;
        o[8] += hi;
      } else {
        __half* o = (EPI == EPI_STORE_OUT ? reinterpret_cast<__half*>(a.step->out) : a.out_h) +
                    (int64_t)tok * a.ldo + mt * 16 + g;
        o[0] = __float2half_rn(lo);
        o[8] = __float2half_rn(hi);
      }
    }
  }
}

template <int NT, int WFMT, int XMODE, int EPI>
cudaError_t launch_t(const Launch& L, const GemvArgs& a) {
  dim3 grid((a.n_mtiles + a.mpc - 1) / a.mpc, a.ks);
  dim3 block(32 * a.mpc * a.wk);
  size_t smem = gemv_smem_bytes(a, NT);
  auto kern = gemv_kernel<NT, WFMT, XMODE, EPI>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.counter) ++*L.counter;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

size_t gemv_smem_bytes(const GemvArgs& a, int) {
  size_t xs = (size_t)a.batch * (a.chunks_per_cta * 64 + 8) * 2;
  size_t red = a.wk > 1 ? (size_t)(a.wk - 1) * a.mpc * 32 * 8 * 4 : 0;
  size_t misc = (size_t)(9 * MAG_MAX_BATCH) * 4;
  size_t body = xs > red ? xs : red;
  return ((body + 15) / 16) * 16 + misc;
}

cudaError_t launch_gemv(const Launch& L, const GemvArgs& a, int wfmt, int xmode, int epi) {
  const bool two = a.batch > 8;
#define MAG_GEMV_CASE(NT_, W_, X_, E_) \
  if ((NT_ == 2) == two && wfmt == W_ && xmode == X_ && epi == E_) return launch_t<NT_, W_, X_, E_>(L, a);
#define MAG_GEMV_NT(W_, X_, E_) MAG_GEMV_CASE(1, W_, X_, E_) MAG_GEMV_CASE(2, W_, X_, E_)
  MAG_GEMV_NT(W_W4, X_NORM, EPI_STORE)
  MAG_GEMV_NT(W_W4, X_F16, EPI_STORE)
  MAG_GEMV_NT(W_W4, X_F16, EPI_RESID)
  MAG_GEMV_NT(W_W4, X_NORM, EPI_SWIGLU)
  MAG_GEMV_NT(W_W4, X_F16, EPI_SWIGLU)
  MAG_GEMV_NT(W_F16, X_NORM, EPI_STORE_OUT)
  MAG_GEMV_NT(W_F16, X_F16, EPI_STORE_OUT)
#undef MAG_GEMV_NT
#undef MAG_GEMV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace mag
