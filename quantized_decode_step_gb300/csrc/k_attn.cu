// KV side of the decode step: RoPE + KV append into the block pool, bulk KV
// store, and split-K flash-decode GQA attention over the pool.
//
// Pool ("5. Core modules" 5.2: a preallocated KV pool; 5.4: FP16 / INT8 /
// INT4 KV): 16-token blocks; the bytes of (layer, block) hold K data
// [Hkv][16][d], V data, K meta [Hkv][16], V meta. INT8 keeps one fp16 scale
// per (token, head) (s = fp16(max|x|/127), q = rint(x/s) clamped to +-127);
// INT4 keeps the 4-bit group-32 codes of head_dim with fp16 (scale, min) per
// group.
//
// Attention: each block of the grid owns one (session, KV head, split) and
// the G query heads that read that KV head. QK^T and PV run on m16n8k16
// tensor-core MMAs (fp16 in, fp32 accumulate) with the query heads as the M
// rows (padded to 16), keys/values converted to fp16 in registers (INT8 codes
// are exact small integers whose scale is folded into the scores and the
// probabilities; INT4 codes are dequantised with scale and min). The softmax
// is the online (running-max) form, in exp2 with log2(e) folded into the
// score scale. Split partials (m, l, o) are merged in split order by the
// last block of each (session, KV head) to arrive.
#include "kernels.h"

namespace mag {

namespace {

// ---------------------------------------------------------------- store of one (token, head) vector
// x: the d fp16 values in shared memory. Called by every thread of the block;
// thread i < d owns element i and warp w < d/32 owns elements 32w..32w+31
// (one INT4 group). The quantisers take their decisions in fp32 with IEEE
// division and round-half-even, group minima and maxima in index order, so
// the stored bytes are fixed by the rule alone.
__device__ void store_vec(const PoolGeom& P, int layer, int blk, int slot, int head, int which, const __half* x,
                          float* red) {
  const int i = threadIdx.x, lane = i & 31, w = i >> 5, d = P.head_dim;
  const bool act = i < d;  // whole warps: d % 32 == 0
  uint8_t* data = pool_vec(P, layer, blk, which, head, slot);
  const float xi = act ? __half2float(x[i]) : 0.f;
  if (P.kv_dtype == 0) {
    if (act) reinterpret_cast<__half*>(data)[i] = x[i];
  } else if (P.kv_dtype == 1) {
    if (act) {
      const float a = warp_max(fabsf(xi));
      if (lane == 0) red[w] = a;
    }
    __syncthreads();
    if (act) {
      float amax = red[0];
      for (int j = 1; j < d / 32; ++j) amax = fmaxf(amax, red[j]);
      const __half s16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
      const float s = __half2float(s16);
      int q = 0;
      if (s != 0.0f) {
        q = (int)rintf(__fdiv_rn(xi, s));
        q = max(-127, min(127, q));
      }
      reinterpret_cast<int8_t*>(data)[i] = (int8_t)q;
      if (i == 0) *reinterpret_cast<__half*>(pool_vec(P, layer, blk, 2 + which, head, slot)) = s16;
    }
    __syncthreads();  // red reused by the next call
  } else if (act) {
    float lo = 0.f, hi = 0.f;
    if (lane == 0) {
      lo = hi = __half2float(x[32 * w]);
      for (int j = 1; j < 32; ++j) {
        const float v = __half2float(x[32 * w + j]);
        if (v < lo) lo = v;
        if (v > hi) hi = v;
      }
    }
    lo = __shfl_sync(0xffffffffu, lo, 0);
    hi = __shfl_sync(0xffffffffu, hi, 0);
    const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.0f));
    const __half m16 = __float2half_rn(lo);
    const float s = __half2float(s16), m = __half2float(m16);
    int q = 0;
    if (s != 0.0f) {
      q = (int)rintf(__fdiv_rn(__fsub_rn(xi, m), s));
      q = max(0, min(15, q));
    }
    const int qn = __shfl_down_sync(0xffffffffu, q, 1);
    if ((lane & 1) == 0) data[i >> 1] = (uint8_t)(q | (qn << 4));
    if (lane == 0) {
      __half2* meta = reinterpret_cast<__half2*>(pool_vec(P, layer, blk, 2 + which, head, slot));
      meta[w] = __halves2half2(s16, m16);
    }
  }
}

// ---------------------------------------------------------------- bulk store of given (rotated) K/V
__global__ void kv_store_kernel(const KvStoreArgs a) {
  __shared__ __half xk[128], xv[128];
  __shared__ float red[8];
  const int t = blockIdx.x, h = blockIdx.y, l = blockIdx.z, i = threadIdx.x;
  const int H = a.pool.n_kv_heads, d = a.pool.head_dim;
  const int64_t src = (((int64_t)l * a.n_tok + t) * H + h) * d;
  xk[i] = a.k[src + i];
  xv[i] = a.v[src + i];
  __syncthreads();
  const int pos = a.pos0 + t;
  const int blk = a.table[pos >> 4];
  store_vec(a.pool, l, blk, pos & 15, h, 0, xk, red);
  store_vec(a.pool, l, blk, pos & 15, h, 1, xv, red);
}

// ---------------------------------------------------------------- KV element conversion to fp16 pairs
// 4 signed bytes -> 2 half2 of exact integers, natural order.
__device__ __forceinline__ void i8x4_to_h2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const __half2 k1152 = __float2half2_rn(1152.0f);
  uint32_t u = w ^ 0x80808080u;
  lo = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4140)), k1152));
  hi = h2_as_u32(__hsub2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4342)), k1152));
}

// 8 nibbles (k0 in bits 0-3 ... k7 in bits 28-31) -> (k0,k4) (k1,k5) (k2,k6) (k3,k7) as s*q + m.
__device__ __forceinline__ uint4 u4x8_to_h2(uint32_t w, __half2 sm) {
  const __half2 k1024 = __float2half2_rn(1024.0f);
  const __half2 k1_16 = __float2half2_rn(0.0625f);
  const __half2 km64 = __float2half2_rn(-64.0f);
  __half2 s2 = __low2half2(sm), m2 = __high2half2(sm);
  uint32_t w2 = w >> 8;
  uint4 o;
  o.x = h2_as_u32(__hfma2(__hsub2(u32_as_h2(lop3_and_or(w, 0x000F000Fu, 0x64006400u)), k1024), s2, m2));
  o.y = h2_as_u32(__hfma2(__hfma2(u32_as_h2(lop3_and_or(w, 0x00F000F0u, 0x64006400u)), k1_16, km64), s2, m2));
  o.z = h2_as_u32(__hfma2(__hsub2(u32_as_h2(lop3_and_or(w2, 0x000F000Fu, 0x64006400u)), k1024), s2, m2));
  o.w = h2_as_u32(__hfma2(__hfma2(u32_as_h2(lop3_and_or(w2, 0x00F000F0u, 0x64006400u)), k1_16, km64), s2, m2));
  return o;
}

__device__ __forceinline__ uint4 perm_k0k4(uint4 v) {
  uint4 o;
  o.x = __byte_perm(v.x, v.z, 0x5410);
  o.y = __byte_perm(v.x, v.z, 0x7632);
  o.z = __byte_perm(v.y, v.w, 0x5410);
  o.w = __byte_perm(v.y, v.w, 0x7632);
  return o;
}

// dim offset of V slot n within a lane's dims (INT4 nibble order, identity otherwise)
template <int DT>
__device__ __forceinline__ int v_slot_dim(int n) {
  if (DT != 2) return n;
  return (n & 8) + ((n & 7) >> 1) + 4 * (n & 1);
}

// K slab (32 dims) of one token for lane t: 4 half2 = b0/b1 of k-steps 2s and 2s+1.
template <int DT>
__device__ __forceinline__ uint4 load_k_slab(const PoolGeom& P, const uint8_t* row, const uint8_t* meta, int s, int t) {
  if (DT == 0) return *reinterpret_cast<const uint4*>(row + (32 * s + 8 * t) * 2);
  if (DT == 1) {
    uint2 w = *reinterpret_cast<const uint2*>(row + 32 * s + 8 * t);
    uint4 o;
    i8x4_to_h2(w.x, o.x, o.y);
    i8x4_to_h2(w.y, o.z, o.w);
    return o;
  }
  uint32_t w = *reinterpret_cast<const uint32_t*>(row + 16 * s + 4 * t);
  __half2 sm = *reinterpret_cast<const __half2*>(meta + 4 * s);
  return u4x8_to_h2(w, sm);
}

// V dims of lane group gi for one token: NV halves as NV/2 words, slot order.
template <int D, int DT>
__device__ __forceinline__ void load_v_row(const uint8_t* row, const uint8_t* meta, int gi, uint32_t (&out)[D / 16]) {
  constexpr int NV = D / 8;
  if (DT == 0) {
    const uint4* p = reinterpret_cast<const uint4*>(row + gi * NV * 2);
#pragma unroll
    for (int j = 0; j < NV / 8; ++j) {
      uint4 v = p[j];
      out[4 * j + 0] = v.x;
      out[4 * j + 1] = v.y;
      out[4 * j + 2] = v.z;
      out[4 * j + 3] = v.w;
    }
  } else if (DT == 1) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(row + gi * NV);
#pragma unroll
    for (int j = 0; j < NV / 4; ++j) i8x4_to_h2(p[j], out[2 * j], out[2 * j + 1]);
  } else {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(row + gi * NV / 2);
    __half2 sm = *reinterpret_cast<const __half2*>(meta + 4 * ((gi * NV) / 32));
#pragma unroll
    for (int j = 0; j < NV / 8; ++j) {
      uint4 o = u4x8_to_h2(p[j], sm);
      out[4 * j + 0] = o.x;
      out[4 * j + 1] = o.y;
      out[4 * j + 2] = o.z;
      out[4 * j + 3] = o.w;
    }
  }
}

__device__ __forceinline__ uint32_t pair_tokens(const uint32_t* ra, const uint32_t* rb, int n) {
  return __byte_perm(ra[n >> 1], rb[n >> 1], (n & 1) ? 0x7632 : 0x5410);
}

// 8 codes of a word as exact fp16 integers in (k0,k4) (k1,k5) (k2,k6) (k3,k7) order.
__device__ __forceinline__ uint4 u4x8_codes(uint32_t w) {
  const __half2 k1024 = __float2half2_rn(1024.0f);
  const __half2 k1_16 = __float2half2_rn(0.0625f);
  const __half2 km64 = __float2half2_rn(-64.0f);
  const uint32_t w2 = w >> 8;
  uint4 o;
  o.x = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(w, 0x000F000Fu, 0x64006400u)), k1024));
  o.y = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w, 0x00F000F0u, 0x64006400u)), k1_16, km64));
  o.z = h2_as_u32(__hsub2(u32_as_h2(lop3_and_or(w2, 0x000F000Fu, 0x64006400u)), k1024));
  o.w = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w2, 0x00F000F0u, 0x64006400u)), k1_16, km64));
  return o;
}

template <int D, int DT>
__global__ void __launch_bounds__(128) attn_kernel(const AttnArgs a) {
  constexpr int NS = D / 32;  // 32-dim slabs of K (one INT4 group each)
  constexpr int NV = D / 8;   // V n-tiles
  constexpr int NW = D / 16;  // words per V row of a lane
  __shared__ float s_m[4][8], s_l[4][8];
  __shared__ float s_acc[4][8][D];
  __shared__ __half s_kv[2][D];
  __shared__ float s_red[8];
  __shared__ float s_cm[64][8], s_cl[64][8];
  __shared__ int s_last;

  const int split = blockIdx.x, gk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gi = lane >> 2, t = lane & 3;
  const int Hq = a.n_heads, Hkv = a.n_kv_heads, G = Hq / Hkv;
  pdl_wait();
  pdl_trigger();
  const int pos = a.step->pos[b], sess = a.step->sess[b];
  const int n_keys = pos + 1;
  const int n_blocks = (n_keys + 15) >> 4;
  const int s_eff = max(1, min(a.n_split, (n_blocks + 3) >> 2));
  const int bps = (n_blocks + s_eff - 1) / s_eff;
  const int blk0 = split * bps, blk1 = min(blk0 + bps, n_blocks);
  const int32_t* table = a.pool.tables + (int64_t)sess * a.pool.table_stride;
  const __half* qkv = a.qkv + (int64_t)b * a.qkv_ld;
  const int64_t pbase = (((int64_t)b * Hkv + gk) * a.n_split + split) * G;

  // the block that holds the new token first appends its K (rotated) and V to the pool
  if (blk0 <= (pos >> 4) && (pos >> 4) < blk1) {
    if (tid < D) {
      s_kv[0][tid] = qkv[(int64_t)(Hq + gk) * D + tid];
      s_kv[1][tid] = qkv[(int64_t)(Hq + Hkv + gk) * D + tid];
    }
    __syncthreads();
    const int phys = table[pos >> 4];
    store_vec(a.pool, a.layer, phys, pos & 15, gk, 0, s_kv[0], s_red);
    store_vec(a.pool, a.layer, phys, pos & 15, gk, 1, s_kv[1], s_red);
    __threadfence_block();
    __syncthreads();
  }

  if (blk0 < blk1) {
    // query fragments: rows = the G heads of this KV head, padded to 16 with zeros
    uint32_t qa[2 * NS][2];
    float qsum[NS];  // INT4: per 32-dim slab, the sum of this row's query values
    const bool hv = gi < G;
    const __half* qrow = qkv + (int64_t)(gk * G + (hv ? gi : 0)) * D;
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      uint4 v = hv ? *reinterpret_cast<const uint4*>(qrow + 32 * s + 8 * t) : make_uint4(0, 0, 0, 0);
      if (DT == 2) {
        const __half* h = reinterpret_cast<const __half*>(&v);
        float sum = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) sum += __half2float(h[e]);
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        qsum[s] = sum;
        v = perm_k0k4(v);
      }
      qa[2 * s][0] = v.x;
      qa[2 * s][1] = v.y;
      qa[2 * s + 1][0] = v.z;
      qa[2 * s + 1][1] = v.w;
    }
    const float sc = 1.4426950408889634f / sqrtf((float)D);  // log2(e) / sqrt(d)
    float m_run = -INFINITY, l_part = 0.f;
    float acc[NV][4];
#pragma unroll
    for (int n = 0; n < NV; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

    for (int blk = blk0 + warp; blk < blk1; blk += 4) {
      const int phys = table[blk];
      // ---- scores S[head][token] of the block's 16 tokens (two n-tiles of 8)
      float sfr[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sfr[nt][0] = sfr[nt][1] = sfr[nt][2] = sfr[nt][3] = 0.f;
        const uint8_t* krow = pool_vec(a.pool, a.layer, phys, 0, gk, gi + 8 * nt);
        if (DT == 2) {
          const uint8_t* kmeta0 = pool_vec(a.pool, a.layer, phys, 2, gk, 8 * nt + 2 * t);
#pragma unroll
          for (int s = 0; s < NS; ++s) {
            const uint4 kq = u4x8_codes(*reinterpret_cast<const uint32_t*>(krow + 16 * s + 4 * t));
            float as[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(as, qa[2 * s][0], 0u, qa[2 * s][1], 0u, kq.x, kq.y);
            mma_16816(as, qa[2 * s + 1][0], 0u, qa[2 * s + 1][1], 0u, kq.z, kq.w);
            // per (token, group): score += s * (q . codes) + m * sum(q)
            const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(kmeta0 + 4 * s));
            const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(kmeta0 + a.pool.meta_bytes + 4 * s));
            sfr[nt][0] = fmaf(f0.x, as[0], fmaf(f0.y, qsum[s], sfr[nt][0]));
            sfr[nt][1] = fmaf(f1.x, as[1], fmaf(f1.y, qsum[s], sfr[nt][1]));
          }
        } else {
#pragma unroll
          for (int s = 0; s < NS; ++s) {
            uint4 kb;
            if (DT == 0) {
              kb = *reinterpret_cast<const uint4*>(krow + (32 * s + 8 * t) * 2);
            } else {
              const uint2 w = *reinterpret_cast<const uint2*>(krow + 32 * s + 8 * t);
              i8x4_to_h2(w.x, kb.x, kb.y);
              i8x4_to_h2(w.y, kb.z, kb.w);
            }
            mma_16816(sfr[nt], qa[2 * s][0], 0u, qa[2 * s][1], 0u, kb.x, kb.y);
            mma_16816(sfr[nt], qa[2 * s + 1][0], 0u, qa[2 * s + 1][1], 0u, kb.z, kb.w);
          }
        }
      }
      // this lane's tokens: (nt, j) -> 16 blk + 8 nt + 2 t + j
      float ks[2][2] = {{1.f, 1.f}, {1.f, 1.f}}, vsc[2][2] = {{1.f, 1.f}, {1.f, 1.f}};
      if (DT == 1) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const __half2 k2 = *reinterpret_cast<const __half2*>(pool_vec(a.pool, a.layer, phys, 2, gk, 8 * nt + 2 * t));
          const __half2 v2 = *reinterpret_cast<const __half2*>(pool_vec(a.pool, a.layer, phys, 3, gk, 8 * nt + 2 * t));
          ks[nt][0] = __low2float(k2);
          ks[nt][1] = __high2float(k2);
          vsc[nt][0] = __low2float(v2);
          vsc[nt][1] = __high2float(v2);
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int tok = blk * 16 + 8 * nt + 2 * t + j;
          float v = sfr[nt][j] * ks[nt][j] * sc;
          v = tok < n_keys ? v : -INFINITY;
          sfr[nt][j] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float corr = exp2f(m_run - m_new);
      m_run = m_new;
      float p[2][2];
      float psum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          p[nt][j] = exp2f(sfr[nt][j] - m_new);
          psum += p[nt][j];
        }
      l_part = l_part * corr + psum;
#pragma unroll
      for (int n = 0; n < NV; ++n) {
        acc[n][0] *= corr;
        acc[n][1] *= corr;
      }
      // P (times the INT8 value scale) as the A operand, split into fp16 hi + lo so the
      // product carries no fp16 rounding of the probabilities: a0 = tokens (2t, 2t+1),
      // a2 = tokens (8+2t, 9+2t)
      float pv[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) pv[nt][j] = p[nt][j] * vsc[nt][j];
      const __half2 h0 = __floats2half2_rn(pv[0][0], pv[0][1]), h2 = __floats2half2_rn(pv[1][0], pv[1][1]);
      const float2 f0 = __half22float2(h0), f2 = __half22float2(h2);
      const uint32_t pa0 = h2_as_u32(h0), pa2 = h2_as_u32(h2);
      const uint32_t pl0 = h2_as_u32(__floats2half2_rn(pv[0][0] - f0.x, pv[0][1] - f0.y));
      const uint32_t pl2 = h2_as_u32(__floats2half2_rn(pv[1][0] - f2.x, pv[1][1] - f2.y));
      // ---- V rows of tokens 2t, 2t+1, 8+2t, 9+2t
      uint32_t v0[NW], v1[NW], v8[NW], v9[NW];
      load_v_row<D, DT>(pool_vec(a.pool, a.layer, phys, 1, gk, 2 * t),
                        DT == 2 ? pool_vec(a.pool, a.layer, phys, 3, gk, 2 * t) : nullptr, gi, v0);
      load_v_row<D, DT>(pool_vec(a.pool, a.layer, phys, 1, gk, 2 * t + 1),
                        DT == 2 ? pool_vec(a.pool, a.layer, phys, 3, gk, 2 * t + 1) : nullptr, gi, v1);
      load_v_row<D, DT>(pool_vec(a.pool, a.layer, phys, 1, gk, 8 + 2 * t),
                        DT == 2 ? pool_vec(a.pool, a.layer, phys, 3, gk, 8 + 2 * t) : nullptr, gi, v8);
      load_v_row<D, DT>(pool_vec(a.pool, a.layer, phys, 1, gk, 9 + 2 * t),
                        DT == 2 ? pool_vec(a.pool, a.layer, phys, 3, gk, 9 + 2 * t) : nullptr, gi, v9);
#pragma unroll
      for (int n = 0; n < NV; ++n) {
        const uint32_t b0 = pair_tokens(v0, v1, n), b1 = pair_tokens(v8, v9, n);
        mma_16816(acc[n], pa0, 0u, pa2, 0u, b0, b1);
        mma_16816(acc[n], pl0, 0u, pl2, 0u, b0, b1);
      }
    }
    // ---- merge the 4 warps of this block
    float l_tot = l_part;
    l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 1);
    l_tot += __shfl_xor_sync(0xffffffffu, l_tot, 2);
    if (hv) {
      if (t == 0) {
        s_m[warp][gi] = m_run;
        s_l[warp][gi] = l_tot;
      }
#pragma unroll
      for (int n = 0; n < NV; ++n) {
        s_acc[warp][gi][(2 * t) * NV + v_slot_dim<DT>(n)] = acc[n][0];
        s_acc[warp][gi][(2 * t + 1) * NV + v_slot_dim<DT>(n)] = acc[n][1];
      }
    }
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += blockDim.x) {
      const int h = idx / D, dim = idx - h * D;
      float mm = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) mm = fmaxf(mm, s_m[w][h]);
      float o = 0.f, l = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float e = exp2f(s_m[w][h] - mm);  // warps without blocks: m = -inf -> 0
        o += s_acc[w][h][dim] * e;
        l += s_l[w][h] * e;
      }
      a.part_o[(pbase + h) * D + dim] = o;
      if (dim == 0) {
        a.part_ml[(pbase + h) * 2 + 0] = mm;
        a.part_ml[(pbase + h) * 2 + 1] = l;
      }
    }
  }
  // ---- the last block of this (session, KV head) merges the splits in order
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.counters + (int64_t)b * Hkv + gk, 1u) == (unsigned)(a.n_split - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int n_valid = (n_blocks + bps - 1) / bps;  // splits that hold blocks
  const int64_t base0 = (((int64_t)b * Hkv + gk) * a.n_split) * G;
  for (int i = tid; i < n_valid * G; i += blockDim.x) {
    const int s = i / G, h = i - s * G;
    s_cm[s][h] = __ldcg(a.part_ml + (base0 + i) * 2);
    s_cl[s][h] = __ldcg(a.part_ml + (base0 + i) * 2 + 1);
  }
  __syncthreads();
  if (tid < G) {
    float mm = -INFINITY;
    for (int s = 0; s < n_valid; ++s) mm = fmaxf(mm, s_cm[s][tid]);
    float l = 0.f;
    for (int s = 0; s < n_valid; ++s) l += s_cl[s][tid] * exp2f(s_cm[s][tid] - mm);
    const float inv = 1.0f / l;
    for (int s = 0; s < n_valid; ++s) s_cm[s][tid] = exp2f(s_cm[s][tid] - mm) * inv;  // split weights
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += blockDim.x) {
    const int h = idx / D, dim = idx - h * D;
    const float* po = a.part_o + (base0 + h) * D + dim;
    float o = 0.f;
#pragma unroll 8
    for (int s = 0; s < n_valid; ++s) o += __ldcg(po + (int64_t)s * G * D) * s_cm[s][h];
    a.o[(int64_t)b * a.ldo + (int64_t)(gk * G + h) * D + dim] = __float2half_rn(o);
  }
  if (tid == 0) a.counters[(int64_t)b * Hkv + gk] = 0;
}

template <typename K, typename Args>
cudaError_t launch_ex(const Launch& L, K kern, dim3 grid, dim3 block, size_t smem, const Args& a) {
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

cudaError_t launch_kv_store(const Launch& L, const KvStoreArgs& a) {
  if (a.n_tok == 0) return cudaSuccess;
  return launch_ex(L, kv_store_kernel, dim3(a.n_tok, a.pool.n_kv_heads, a.n_layers), dim3(a.pool.head_dim), 0, a);
}

cudaError_t launch_attention(const Launch& L, const AttnArgs& a, int batch) {
  dim3 grid(a.n_split, a.n_kv_heads, batch), block(128);
  const int dt = a.pool.kv_dtype;
  if (a.head_dim == 128) {
    if (dt == 0) return launch_ex(L, attn_kernel<128, 0>, grid, block, 0, a);
    if (dt == 1) return launch_ex(L, attn_kernel<128, 1>, grid, block, 0, a);
    return launch_ex(L, attn_kernel<128, 2>, grid, block, 0, a);
  }
  if (a.head_dim == 64) {
    if (dt == 0) return launch_ex(L, attn_kernel<64, 0>, grid, block, 0, a);
    if (dt == 1) return launch_ex(L, attn_kernel<64, 1>, grid, block, 0, a);
    return launch_ex(L, attn_kernel<64, 2>, grid, block, 0, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mag
