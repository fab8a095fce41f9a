// W4A16 (and fp16) matrix-vector products of the decode step on mma.sync.
//
// y[b][n] = sum_k deq(W)[n][k] x[b][k] for a handful of tokens b, with the
// weights streamed once from HBM in the packed 4-bit group-32 layout the
// library takes at load time ("5. Core modules" 5.1: 4-bit weights, FP16
// activations). No repacking. Per 64-wide k-chunk a lane reads, for rows g
// and g+8 of its 16-row tile, one 32-bit word of each of the chunk's two
// groups, turns its 8 nibbles into exact small integers in fp16 with a LOP3
// into the mantissa of 1024 (the int4-to-fp16 conversion of Kim et al., "Who
// Says Elephants Can't Run", 2022) and feeds m16n8k16 tensor-core MMAs with
// fp32 accumulators, one fresh accumulator per group. Scale and min are
// applied per group in fp32:
//     sum_k (s q_k + m) x_k = s * sum_k q_k x_k + m * X_g,   X_g = sum_{k in g} x_k,
// so the result carries no rounding of the dequantised weights; the group
// sums X_g come with the activations from their producer. The activations are
// stored in 8-wide units in the order (x0,x4,x1,x5,x2,x6,x3,x7), which is the
// k order the nibble pairs come out in, so a lane's B fragments for one group
// are one 128-bit load.
//
// Epilogues fused around the product:
//   QKV      fp16 q/k/v, q and k rotated (RoPE, pre-generated table) -- the
//            tile's rows g and g+8 are the pair (i, i + d/2) of one head;
//   RESID    fp32 residual add, per-tile sums of squares, and in the last
//            block to finish the RMSNorm of the new residual for the next
//            projection (or the fp16 hidden-state output);
//   SWIGLU   silu(gate) * up of interleaved gate/up rows, with group sums;
//   OUT      fp16 logits into the caller's buffer.
// Weight loads for the first chunks are issued before the programmatic-
// dependent-launch wait, so they overlap the previous kernel's tail.
#include "kernels.h"

namespace mag {

namespace {

constexpr int kStages = 4;

struct W4Stage {
  uint32_t wg0, wg1, wv0, wv1;  // row g / g+8, group 0 / 1 of the chunk: word t
  uint2 sg, sv;                 // (scale, min) of groups 0 and 1, rows g and g+8
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

__device__ __forceinline__ uint32_t ldg_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_nc_u2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ void load_stage(W4Stage& st, const GemvArgs& a, int row_g, int row_g8, int c, int t) {
  const uint8_t* pg = a.w + (int64_t)row_g * a.w_row_bytes + c * 32 + t * 4;
  const uint8_t* pv = a.w + (int64_t)row_g8 * a.w_row_bytes + c * 32 + t * 4;
  const bool g1 = 2 * c + 1 < a.sm_row;  // the chunk's second group exists
  st.wg0 = ldg_stream_u32(pg);
  st.wv0 = ldg_stream_u32(pv);
  st.wg1 = g1 ? ldg_stream_u32(pg + 16) : 0u;
  st.wv1 = g1 ? ldg_stream_u32(pv + 16) : 0u;
  const __half2* sg = a.sm + (int64_t)row_g * a.sm_row + 2 * c;
  const __half2* sv = a.sm + (int64_t)row_g8 * a.sm_row + 2 * c;
  if (g1) {
    st.sg = ldg_nc_u2(sg);
    st.sv = ldg_nc_u2(sv);
  } else {
    st.sg = make_uint2(ldg_nc_u32(sg), 0u);
    st.sv = make_uint2(ldg_nc_u32(sv), 0u);
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

// The 8 codes of a word (k0 in bits 0-3 ... k7 in bits 28-31) as exact fp16
// integers, paired (k0,k4) (k1,k5) (k2,k6) (k3,k7).
struct Q4 {
  uint32_t e0, e1, e2, e3;
};
__device__ __forceinline__ Q4 codes_word(uint32_t w) {
  const __half2 k1024 = __float2half2_rn(1024.0f);
  const __half2 k1_16 = __float2half2_rn(0.0625f);
  const __half2 km64 = __float2half2_rn(-64.0f);
  uint32_t w2 = w >> 8;
  Q4 q;
  q.e0 = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(w, 0x000F000Fu, 0x64006400u)), k1024));
  q.e1 = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w, 0x00F000F0u, 0x64006400u)), k1_16, km64));
  q.e2 = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(w2, 0x000F000Fu, 0x64006400u)), k1024));
  q.e3 = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w2, 0x00F000F0u, 0x64006400u)), k1_16, km64));
  return q;
}

// Activation fragments of one chunk for one 8-token n-tile: W4 -> units 8c+t
// (group 0) and 8c+4+t (group 1); fp16 weights -> units 8c+2t, 8c+2t+1.
struct XFrag {
  uint4 u0, u1;
  float2 s_lo, s_hi;  // W4: group sums (groups 0, 1) of tokens 2t and 2t+1 of the n-tile
};

// acc += scale * (q . x) + min * X_g for rows g (acc[0..1]) and g + 8 (acc[2..3]).
__device__ __forceinline__ void gemv_fma_group(float (&acc)[4], const float (&aq)[4], uint32_t sm_g, uint32_t sm_g8,
                                               float x_lo, float x_hi, bool one_tok) {
  const float2 fg = __half22float2(u32_as_h2(sm_g)), fv = __half22float2(u32_as_h2(sm_g8));
  // fg = (scale, min) of row g, fv of row g + 8; columns: tokens 2t (lo) and 2t+1 (hi)
  acc[0] = fmaf(fg.x, aq[0], fmaf(fg.y, x_lo, acc[0]));
  acc[2] = fmaf(fv.x, aq[2], fmaf(fv.y, x_lo, acc[2]));
  if (!one_tok) {
    acc[1] = fmaf(fg.x, aq[1], fmaf(fg.y, x_hi, acc[1]));
    acc[3] = fmaf(fv.x, aq[3], fmaf(fv.y, x_hi, acc[3]));
  }
}

template <int NT>
__device__ __forceinline__ void compute_stage(const W4Stage& st, float (&acc)[2][4], const XFrag (&xf)[2],
                                              bool one_tok) {
#pragma unroll
  for (int grp = 0; grp < 2; ++grp) {
    const Q4 qg = codes_word(grp ? st.wg1 : st.wg0);
    const Q4 qv = codes_word(grp ? st.wv1 : st.wv0);
    const uint32_t smg = grp ? st.sg.y : st.sg.x, smv = grp ? st.sv.y : st.sv.x;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint4 xb = grp ? xf[nt].u1 : xf[nt].u0;
      float aq[4] = {0.f, 0.f, 0.f, 0.f};
      mma_16816(aq, qg.e0, qv.e0, qg.e1, qv.e1, xb.x, xb.y);
      mma_16816(aq, qg.e2, qv.e2, qg.e3, qv.e3, xb.z, xb.w);
      const float2 xs = grp ? xf[nt].s_hi : xf[nt].s_lo;  // .x token 2t, .y token 2t+1
      gemv_fma_group(acc[nt], aq, smg, smv, xs.x, xs.y, NT == 1 && one_tok);
    }
  }
}

template <int NT>
__device__ __forceinline__ void compute_stage(const F16Stage& st, float (&acc)[2][4], const XFrag (&xf)[2], bool) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    mma_16816(acc[nt], st.g0.x, st.h0.x, st.g0.y, st.h0.y, xf[nt].u0.x, xf[nt].u0.y);
    mma_16816(acc[nt], st.g0.z, st.h0.z, st.g0.w, st.h0.w, xf[nt].u0.z, xf[nt].u0.w);
    mma_16816(acc[nt], st.g1.x, st.h1.x, st.g1.y, st.h1.y, xf[nt].u1.x, xf[nt].u1.y);
    mma_16816(acc[nt], st.g1.z, st.h1.z, st.g1.w, st.h1.w, xf[nt].u1.z, xf[nt].u1.w);
  }
}

// position of element e (0..7) of a unit in the W4 activation order
__device__ __forceinline__ int unit_pos(int e) { return e < 4 ? 2 * e : 2 * (e - 4) + 1; }

template <int NT, int WFMT, int XMODE>
__device__ __forceinline__ void load_x(XFrag (&xf)[2], const GemvArgs& a, const __half* xs_smem, int xrow, int c,
                                       int c_begin, int g, int t) {
  const int B = a.batch;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tok = g + 8 * nt;
    const int ua = WFMT == W_W4 ? 8 * c + t : 8 * c + 2 * t;
    const int ub = WFMT == W_W4 ? 8 * c + 4 + t : 8 * c + 2 * t + 1;
    uint4 u0 = make_uint4(0, 0, 0, 0), u1 = u0;
    if (tok < B) {
      if (XMODE == X_SMEM) {
        const uint4* p = reinterpret_cast<const uint4*>(xs_smem + (size_t)tok * xrow);
        u0 = p[ua - 8 * c_begin];
        u1 = p[ub - 8 * c_begin];
      } else {
        const uint4* p = reinterpret_cast<const uint4*>(a.x + (int64_t)tok * a.ldx);
        if (8 * ua < a.K) u0 = __ldg(p + ua);
        if (8 * ub < a.K) u1 = __ldg(p + ub);
      }
    }
    xf[nt].u0 = u0;
    xf[nt].u1 = u1;
    if (WFMT == W_W4) {
      // group sums for this lane's two C columns (tokens 2t, 2t+1 of the n-tile)
      const int t0 = 8 * nt + 2 * t, t1 = t0 + 1;
      float2 a0 = make_float2(0.f, 0.f), a1 = a0;
      const bool g1 = 2 * c + 1 < a.sm_row;
      if (t0 < B) {
        const float* p = a.xsum + (int64_t)t0 * a.ldxs + 2 * c;
        a0 = g1 ? __ldg(reinterpret_cast<const float2*>(p)) : make_float2(__ldg(p), 0.f);
      }
      if (t1 < B) {
        const float* p = a.xsum + (int64_t)t1 * a.ldxs + 2 * c;
        a1 = g1 ? __ldg(reinterpret_cast<const float2*>(p)) : make_float2(__ldg(p), 0.f);
      }
      xf[nt].s_lo = make_float2(a0.x, a1.x);  // group 0: tokens 2t, 2t+1
      xf[nt].s_hi = make_float2(a0.y, a1.y);  // group 1
    }
  }
}

__device__ __forceinline__ float silu_mul(float gte, float up) { return gte / (1.0f + expf(-gte)) * up; }

// Last block of a residual projection: RMSNorm of the new residual into the
// next projection's fp16 activations (W4 unit order or natural) and their
// group sums, or the fp16 hidden-state output.
__device__ void residual_tail(const GemvArgs& a, float* sm_inv) {
  const int B = a.batch, D = a.n_mtiles * 16, tid = threadIdx.x;
  if (a.tail == TAIL_HIDDEN) {
    __half* out = reinterpret_cast<__half*>(a.step->out);
    for (int i = tid; i < B * D; i += blockDim.x) {
      const int b = i / D, k = i - b * D;
      out[(int64_t)b * D + k] = __float2half_rn(__ldcg(a.r + (int64_t)b * a.ldr + k));
    }
    return;
  }
  if (tid < B) {
    float tot = 0.f;
    for (int m = 0; m < a.n_mtiles; ++m) tot += __ldcg(a.ss_part + (int64_t)m * MAG_MAX_BATCH + tid);
    sm_inv[tid] = 1.0f / sqrtf(tot / (float)D + a.eps);
  }
  __syncthreads();
  const int units = D / 8;  // D % 32 == 0: the 4 units of a group sit in one quad of lanes
  for (int base = 0; base < B * units; base += blockDim.x) {
    const int i = base + tid;
    const bool live = i < B * units;
    const int b = live ? i / units : 0, u = live ? i - b * units : 0;
    float s = 0.f;
    if (live) {
      const float inv = sm_inv[b];
      const float4 r0 = __ldcg(reinterpret_cast<const float4*>(a.r + (int64_t)b * a.ldr + 8 * u));
      const float4 r1 = __ldcg(reinterpret_cast<const float4*>(a.r + (int64_t)b * a.ldr + 8 * u + 4));
      const uint4 gg = *reinterpret_cast<const uint4*>(a.gamma + 8 * u);
      const __half* gh = reinterpret_cast<const __half*>(&gg);
      const float f[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
      __half h[8], o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        h[e] = __float2half_rn(f[e] * inv * __half2float(gh[e]));
        s += __half2float(h[e]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) o[a.xn_permuted ? unit_pos(e) : e] = h[e];
      *reinterpret_cast<uint4*>(a.xn + (int64_t)b * a.ldxn + 8 * u) = *reinterpret_cast<uint4*>(o);
    }
    if (a.xn_sum) {
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (live && (u & 3) == 0) a.xn_sum[(int64_t)b * a.ldxns + u / 4] = s;
    }
  }
}

template <int NT, int WFMT, int XMODE, int EPI>
__global__ void __launch_bounds__(256) gemv_kernel(const GemvArgs a) {
  using Stage = typename StageT<WFMT>::type;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float s_misc[4 * 8 * MAG_MAX_BATCH + MAG_MAX_BATCH];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int mt_local = warp % a.mpc, kw = warp / a.mpc;
  const int mt = blockIdx.x * a.mpc + mt_local;
  const bool mt_ok = mt < a.n_mtiles;
  const int c_begin = blockIdx.y * a.chunks_per_cta;
  const int c_end = min(c_begin + a.chunks_per_cta, a.n_chunks);
  const int n_cc = c_end - c_begin;
  const int B = a.batch;
  const bool one_tok = B == 1;

  int row_g, row_g8;
  if (EPI == EPI_SWIGLU) {
    row_g = mt * 8 + g;
    row_g8 = a.swiglu_f + mt * 8 + g;
  } else if (EPI == EPI_QKV) {
    const int tiles_per_head = a.head_dim / 16, head = mt / tiles_per_head, j = mt - head * tiles_per_head;
    row_g = head * a.head_dim + 8 * j + g;
    row_g8 = row_g + a.head_dim / 2;
  } else {
    row_g = mt * 16 + g;
    row_g8 = row_g + 8;
  }

  const int n_my = (mt_ok && kw < n_cc) ? (n_cc - kw + a.wk - 1) / a.wk : 0;
  Stage st[kStages];
#pragma unroll
  for (int u = 0; u < kStages; ++u)
    if (u < n_my) load_stage(st[u], a, row_g, row_g8, c_begin + kw + u * a.wk, t);

  pdl_wait();
  pdl_trigger();

  const int xrow = n_cc * 64 + 8;  // X_SMEM: halves per staged token row
  const __half* xs = reinterpret_cast<const __half*>(smem);
  if (XMODE == X_SMEM) {
    __half* xw = reinterpret_cast<__half*>(smem);
    const int units = n_cc * 8;
    for (int i = tid; i < units * B; i += blockDim.x) {
      const int b = i / units, u = i - b * units, k = (c_begin * 8 + u) * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (k < a.K) v = *reinterpret_cast<const uint4*>(a.x + (int64_t)b * a.ldx + k);
      *reinterpret_cast<uint4*>(xw + (size_t)b * xrow + u * 8) = v;
    }
    __syncthreads();
  }

  float acc[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;

  for (int i = 0; i < n_my; i += kStages) {
#pragma unroll
    for (int u = 0; u < kStages; ++u) {
      if (i + u < n_my) {
        const Stage cur = st[u];
        const int c = c_begin + kw + (i + u) * a.wk;
        if (i + u + kStages < n_my) load_stage(st[u], a, row_g, row_g8, c + kStages * a.wk, t);
        XFrag xf[2];
        load_x<NT, WFMT, XMODE>(xf, a, xs, xrow, c, c_begin, g, t);
        compute_stage<NT>(cur, acc, xf, one_tok);
      }
    }
  }

  // ---- reduce the wk warps of each m-tile
  if (a.wk > 1) {
    __syncthreads();
    float* red = reinterpret_cast<float*>(smem);
    if (kw > 0 && mt_ok) {
      float* p = red + (((size_t)(kw - 1) * a.mpc + mt_local) * 32 + lane) * 8;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) p[nt * 4 + i] = acc[nt][i];
    }
    __syncthreads();
    if (kw == 0 && mt_ok) {
      for (int w = 1; w < a.wk; ++w) {
        const float* p = red + (((size_t)(w - 1) * a.mpc + mt_local) * 32 + lane) * 8;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[nt][i] += p[nt * 4 + i];
      }
    }
  }

  // ---- reduce across k-split blocks: the last block of the group sums in split order
  if (a.ks > 1) {
    if (kw == 0 && mt_ok) {
      float* p = a.partial + (((size_t)blockIdx.y * a.n_mtiles + mt) * 32 + lane) * (4 * NT);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float4*>(p + nt * 4) = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(a.counters + blockIdx.x, 1u) == (unsigned)(a.ks - 1);
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
          const float4 v = __ldcg(reinterpret_cast<const float4*>(p + nt * 4));
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
  const bool ep = kw == 0 && mt_ok;
  if (EPI == EPI_SWIGLU) {
    // act = silu(gate) * up for rows j = 8 mt + g, stored in W4 unit order, plus group sums
    float gsum[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    if (ep) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int tok = nt * 8 + 2 * t + jj;
          if (tok < B) {
            const __half h = __float2half_rn(silu_mul(acc[nt][jj], acc[nt][jj + 2]));
            a.out_h[(int64_t)tok * a.ldo + 8 * mt + unit_pos(g)] = h;
            gsum[nt][jj] = __half2float(h);
          }
        }
    }
    // sum over the 8 rows of the tile (lanes with equal t), then over the 4 tiles of a group
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        float v = gsum[nt][jj];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        gsum[nt][jj] = v;
      }
    if (kw == 0 && g == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) s_misc[mt_local * MAG_MAX_BATCH + nt * 8 + 2 * t + jj] = gsum[nt][jj];
    }
    __syncthreads();
    // one thread per (group of 4 tiles, token)
    const int n_groups_cta = (a.mpc + 3) / 4;
    for (int i = tid; i < n_groups_cta * B; i += blockDim.x) {
      const int gi = i / B, tok = i - gi * B;
      const int mt0 = blockIdx.x * a.mpc + 4 * gi;
      float s = 0.f;
      for (int m = 0; m < 4; ++m)
        if (4 * gi + m < a.mpc && mt0 + m < a.n_mtiles) s += s_misc[(4 * gi + m) * MAG_MAX_BATCH + tok];
      if (mt0 < a.n_mtiles) a.out_sum[(int64_t)tok * a.ldos + mt0 / 4] = s;
    }
    return;
  }
  if (EPI == EPI_RESID) {
    float ssq[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    if (ep) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int tok = nt * 8 + 2 * t + jj;
          if (tok < B) {
            float* o = a.r + (int64_t)tok * a.ldr + mt * 16 + g;
            const float n0 = o[0] + acc[nt][jj], n1 = o[8] + acc[nt][jj + 2];
            o[0] = n0;
            o[8] = n1;
            ssq[nt][jj] = n0 * n0 + n1 * n1;
          }
        }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        float v = ssq[nt][jj];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        ssq[nt][jj] = v;
      }
    if (ep && g == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int tok = nt * 8 + 2 * t + jj;
          if (tok < B) a.ss_part[(int64_t)mt * MAG_MAX_BATCH + tok] = ssq[nt][jj];
        }
    }
    if (a.tail == TAIL_NONE) return;
    // the last block to finish runs the tail over the whole residual
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(a.counters + gridDim.x, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    residual_tail(a, s_misc);
    if (tid == 0) a.counters[gridDim.x] = 0;
    return;
  }
  if (!ep) return;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int tok = nt * 8 + 2 * t + jj;
      if (tok >= B) continue;
      const float lo = acc[nt][jj], hi = acc[nt][jj + 2];  // rows g and g + 8
      if (EPI == EPI_QKV) {
        // round as the fp16 projection output, then rotate q and k heads: pair (i, i + d/2)
        const float x0 = __half2float(__float2half_rn(lo)), x1 = __half2float(__float2half_rn(hi));
        const int head = row_g / a.head_dim, i = row_g - head * a.head_dim;
        __half* o = a.out_h + (int64_t)tok * a.ldo;
        if (head < a.n_rot_heads) {
          const int pos = a.step->pos[tok], hd = a.head_dim / 2;
          const float c = a.rope_cos[(int64_t)pos * hd + i], s = a.rope_sin[(int64_t)pos * hd + i];
          o[row_g] = __float2half_rn(x0 * c - x1 * s);
          o[row_g8] = __float2half_rn(x0 * s + x1 * c);
        } else {
          o[row_g] = __float2half_rn(lo);
          o[row_g8] = __float2half_rn(hi);
        }
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
  size_t smem = gemv_smem_bytes(a, XMODE);
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

size_t gemv_smem_bytes(const GemvArgs& a, int xmode) {
  size_t xs = xmode == X_SMEM ? (size_t)a.batch * (a.chunks_per_cta * 64 + 8) * 2 : 0;
  size_t red = a.wk > 1 ? (size_t)(a.wk - 1) * a.mpc * 32 * 8 * 4 : 0;
  size_t body = xs > red ? xs : red;
  return ((body + 15) / 16) * 16;
}

cudaError_t launch_gemv(const Launch& L, const GemvArgs& a, int wfmt, int xmode, int epi) {
  const bool two = a.batch > 8;
#define MAG_GEMV_CASE(NT_, W_, X_, E_) \
  if ((NT_ == 2) == two && wfmt == W_ && xmode == X_ && epi == E_) return launch_t<NT_, W_, X_, E_>(L, a);
#define MAG_GEMV_NT(W_, X_, E_) MAG_GEMV_CASE(1, W_, X_, E_) MAG_GEMV_CASE(2, W_, X_, E_)
#define MAG_GEMV_X(W_, E_) MAG_GEMV_CASE(1, W_, X_DIRECT, E_) MAG_GEMV_NT(W_, X_SMEM, E_)
  MAG_GEMV_X(W_W4, EPI_QKV)
  MAG_GEMV_X(W_W4, EPI_RESID)
  MAG_GEMV_X(W_W4, EPI_SWIGLU)
  MAG_GEMV_X(W_F16, EPI_STORE_OUT)
#undef MAG_GEMV_X
#undef MAG_GEMV_NT
#undef MAG_GEMV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace mag
