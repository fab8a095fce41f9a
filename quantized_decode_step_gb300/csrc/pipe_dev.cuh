// Device building blocks of the W4 / fp16 decode GEMV for up to 4 tokens (k_gemv_pipe.cu).
#pragma once
#include "kernels.h"

namespace mag {
namespace pipe {

constexpr int kCWarps = 16;                     // warps per block
constexpr int kThreads = kCWarps * 32;
constexpr int kMaxSlots = 8;                    // ring slots per warp
constexpr uint32_t kSpinLimit = kWaitPolls;     // mbarrier polls before a wait is declared stuck
constexpr float kCodeUnit = 16777216.0f;        // 2^24

template <int WFMT>
struct ChunkFmt;
template <>
struct ChunkFmt<W_W4> {
  static constexpr int kBytes = kTileBytes;  // 512 B codes (lane order) + 128 B (scale, min)
  static constexpr int kPerSlot = 4;         // chunks per ring slot (one bulk copy)
};
template <>
struct ChunkFmt<W_F16> {
  static constexpr int kBytes = 2048;  // 16 rows x 64 k fp16, lane order (64 B per lane)
  static constexpr int kPerSlot = 1;
};
__host__ __device__ constexpr int slot_bytes(int wfmt) { return wfmt == W_W4 ? 4 * kTileBytes : 2048; }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
// One poll: the thread may sleep until the phase completes or up to ~1 us (the suspend-time hint), so that a
// warp waiting for its copy does not take issue slots from the warps that are computing.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of the given parity to complete (at most `limit` polls).
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(b, parity)) return true;
  return false;
}
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// The same on 32-bit shared-memory addresses (the window loop keeps its slot and barrier addresses in
// registers, so that nothing is converted per use).
__device__ __forceinline__ bool mbar_try_wait_a(uint32_t b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(b), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_a(uint32_t b, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait_a(b, parity)) return true;
  return false;
}
// Arm the barrier for `bytes` and copy them, in the lanes where `on` is set (no branch around it).
__device__ __forceinline__ void bulk_copy_a(bool on, uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "setp.ne.u32 q, %4, 0;\n\t"
      "@q mbarrier.arrive.expect_tx.shared::cta.b64 _, [%3], %2;\n\t"
      "@q cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "r"((uint32_t)on)
      : "memory");
}

// D = A * B (fp16 in, fp32 out) with a zero accumulator.
__device__ __forceinline__ void mma_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                      uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// Layout of the dynamic shared memory of one block.
struct PipeSmem {
  uint32_t full, ring, x, xs, part, tcnt, bounds, red, zero, total;
};
__host__ __device__ inline PipeSmem pipe_smem(int wfmt, int B, int n_chunks, int slots, int t_max) {
  PipeSmem L;
  const uint32_t xrow = n_chunks * 64 + 8;  // halves per token row (+8: spreads the rows over the banks)
  const uint32_t grow = 2 * n_chunks + 2;   // group sums per token row
  L.full = 0;                               // [warp][kMaxSlots] mbarriers
  L.ring = kCWarps * kMaxSlots * 8;         // [warp][slots][slot bytes]
  L.x = L.ring + (uint32_t)kCWarps * slots * slot_bytes(wfmt);
  L.xs = L.x + ((B * xrow * 2 + 15) & ~15u);
  L.part = L.xs + ((B * grow * 4 + 15) & ~15u);  // [warp][first / last tile][lane] float4
  L.tcnt = L.part + kCWarps * 2 * 32 * 16;  // per tile: warps done with their part
  L.bounds = L.tcnt + ((uint32_t)t_max * 4 + 15) / 16 * 16;  // first pair of every warp's run, and the end
  L.red = L.bounds + (kCWarps + 1 + 3) / 4 * 16;
  L.zero = L.red + (kCWarps + 1) * MAG_MAX_BATCH * 4;  // 16 zero bytes
  L.total = L.zero + 16;
  return L;
}

// Stage the activations of all K into shared memory. W4: units of 8 in the
// order (x0,x4,x2,x6, x1/16,x5/16,x3/16,x7/16) with the group sums of the
// unscaled values; fp16: natural order. XSRC_RESID: x = fp16(r / sqrt(mean(r^2)
// + eps) * gamma), the mean over this block's own pass over r.
template <int WFMT, int XSRC, int B, typename Hook>
__device__ void stage_x(const GemvArgs& a, __half* xw, float* xsw, float* red, uint32_t xrow, uint32_t grow,
                        Hook after_loads) {
  constexpr int NT = kCWarps * 32;
  // units of 8 values a thread loads ahead into registers (all of them for D = 4096, and for FFN 14336 at one
  // token); the hook runs once their loads are issued, so that what it queues comes after them
  constexpr int KR = XSRC == XSRC_F16 ? 4 : B;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int upt = a.n_chunks * 8;  // 8-value units per token row
  const int U = B * upt;
  const int n_iter = (U + NT - 1) / NT;  // the same for every thread
  float rv[KR][8];
  uint4 hv[KR];  // XSRC_F16: the activations; XSRC_RESID: the gains
  auto load = [&](int u, float (&v)[8], uint4& h) {
    const int b = u / upt, k = (u - b * upt) * 8;
    const bool ok = u < U && k < a.K;
    if (XSRC == XSRC_RESID) {
      if (ok) {
        const float4 r0 = __ldcg(reinterpret_cast<const float4*>(a.r + (int64_t)b * a.ldr + k));
        const float4 r1 = __ldcg(reinterpret_cast<const float4*>(a.r + (int64_t)b * a.ldr + k + 4));
        v[0] = r0.x, v[1] = r0.y, v[2] = r0.z, v[3] = r0.w, v[4] = r1.x, v[5] = r1.y, v[6] = r1.z, v[7] = r1.w;
        h = *reinterpret_cast<const uint4*>(a.gamma + k);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
        h = make_uint4(0, 0, 0, 0);
      }
    } else {
      // L2 only: the activations may have been written by another block of the same (persistent) kernel
      h = ok ? __ldcg(reinterpret_cast<const uint4*>(a.x + (int64_t)b * a.ldx + k)) : make_uint4(0, 0, 0, 0);
    }
  };
#pragma unroll
  for (int i = 0; i < KR; ++i)
    if (i < n_iter) load(tid + i * NT, rv[i], hv[i]);
  after_loads();

  float inv[B];
  if (XSRC == XSRC_RESID) {
    float ss[B];
#pragma unroll
    for (int b = 0; b < B; ++b) ss[b] = 0.f;
    auto add_sq = [&](int u, const float (&v)[8]) {
      const int b = u / upt;
      float sq = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) sq = fmaf(v[e], v[e], sq);
#pragma unroll
      for (int bb = 0; bb < B; ++bb) ss[bb] += bb == b ? sq : 0.f;
    };
#pragma unroll
    for (int i = 0; i < KR; ++i)
      if (i < n_iter) add_sq(tid + i * NT, rv[i]);
    for (int i = KR; i < n_iter; ++i) {
      float v[8];
      uint4 h;
      load(tid + i * NT, v, h);
      add_sq(tid + i * NT, v);
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const float s = warp_sum(ss[b]);
      if (lane == 0) red[warp * MAG_MAX_BATCH + b] = s;
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < B; ++b) {
      float tot = 0.f;
      for (int w = 0; w < kCWarps; ++w) tot += red[w * MAG_MAX_BATCH + b];
      inv[b] = 1.0f / sqrtf(tot / (float)a.K + a.eps);
    }
  }
  // write unit u from its loaded values
  auto put = [&](int u, const float (&v)[8], const uint4 hin) {
    const bool live = u < U;
    const int b = live ? u / upt : 0, ul = live ? u - b * upt : 0, k = ul * 8;
    float s = 0.f;
    if (live) {
      __half h[8];
      if (k >= a.K) {
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(0.f);
      } else if (XSRC == XSRC_F16) {
        *reinterpret_cast<uint4*>(h) = hin;
      } else {
        float ib = inv[0];
#pragma unroll
        for (int bb = 1; bb < B; ++bb) ib = bb == b ? inv[bb] : ib;
        const __half* gh = reinterpret_cast<const __half*>(&hin);
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(v[e] * ib * __half2float(gh[e]));
      }
      __half o[8];
      if (WFMT == W_W4) {
        const __half k16 = __float2half_rn(0.0625f);
        o[0] = h[0], o[1] = h[4], o[2] = h[2], o[3] = h[6];
        o[4] = __hmul(h[1], k16), o[5] = __hmul(h[5], k16), o[6] = __hmul(h[3], k16), o[7] = __hmul(h[7], k16);
#pragma unroll
        for (int e = 0; e < 8; ++e) s += __half2float(h[e]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = h[e];
      }
      *reinterpret_cast<uint4*>(xw + (size_t)b * xrow + 8 * ul) = *reinterpret_cast<uint4*>(o);
    }
    if (WFMT == W_W4) {
      // the 4 units of a 32-wide group sit in one quad of lanes (units per row are a multiple of 4)
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (live && (ul & 3) == 0) xsw[(size_t)b * grow + ul / 4] = s;
    }
  };
#pragma unroll
  for (int i = 0; i < KR; ++i)
    if (i < n_iter) put(tid + i * NT, rv[i], hv[i]);
  for (int i = KR; i < n_iter; ++i) {
    float v[8];
    uint4 h;
    load(tid + i * NT, v, h);
    put(tid + i * NT, v, h);
  }
  __syncthreads();
}

// One W4 chunk: lane (g, t) holds words t of rows g and g+8 for the chunk's two groups and their (scale, min).
// acc[0..3]: scale * codes.x in units of 2^-24 for (row g, token 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1);
// acc[4..7]: min * X_g for the same.
template <int B>
__device__ __forceinline__ void w4_chunk(const uint4 cw, const uint4 sm, const uint4 xa, const uint4 xb,
                                         const float2 X0, const float2 X1, float (&acc)[8]) {
#pragma unroll
  for (int grp = 0; grp < 2; ++grp) {
    const uint32_t wg = grp ? cw.y : cw.x, wv = grp ? cw.w : cw.z;
    const uint32_t sg = wg >> 8, sv = wv >> 8;
    const uint4 xu = grp ? xb : xa;
    float d[4];
    mma_z(d, wg & 0x000F000Fu, wv & 0x000F000Fu, sg & 0x000F000Fu, sv & 0x000F000Fu, xu.x, xu.y);
    mma_16816(d, wg & 0x00F000F0u, wv & 0x00F000F0u, sg & 0x00F000F0u, sv & 0x00F000F0u, xu.z, xu.w);
    const float2 fg = __half22float2(u32_as_h2(grp ? sm.y : sm.x));
    const float2 fv = __half22float2(u32_as_h2(grp ? sm.w : sm.z));
    const float x0 = grp ? X0.y : X0.x;
    acc[0] = fmaf(fg.x, d[0], acc[0]);
    acc[2] = fmaf(fv.x, d[2], acc[2]);
    acc[4] = fmaf(fg.y, x0, acc[4]);
    acc[6] = fmaf(fv.y, x0, acc[6]);
    if (B > 1) {
      const float x1 = grp ? X1.y : X1.x;
      acc[1] = fmaf(fg.x, d[1], acc[1]);
      acc[3] = fmaf(fv.x, d[3], acc[3]);
      acc[5] = fmaf(fg.y, x1, acc[5]);
      acc[7] = fmaf(fv.y, x1, acc[7]);
    }
  }
}

__device__ __forceinline__ float silu_mul(float gte, float up) { return gte / (1.0f + expf(-gte)) * up; }

// The epilogue of tile mt for lane (g, t): v = (row g, token 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1).
template <int EPI, int B>
__device__ __forceinline__ void tile_epilogue(const GemvArgs& a, int mt, const float4 v, int g, int t) {
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const int tok = 2 * t + jj;
    if (tok >= B) continue;
    const float lo = jj ? v.y : v.x, hi = jj ? v.w : v.z;  // rows g and g + 8 of the tile
    if (EPI == EPI_RESID) {
      float* o = a.r + (int64_t)tok * a.ldr + mt * 16 + g;
      o[0] = __ldcg(o) + lo;
      o[8] = __ldcg(o + 8) + hi;
    } else if (EPI == EPI_STORE_OUT) {
      __half* o = reinterpret_cast<__half*>(a.step->out) + (int64_t)tok * a.ldo + mt * 16 + g;
      o[0] = __float2half_rn(lo);
      o[8] = __float2half_rn(hi);
    } else if (EPI == EPI_SWIGLU) {
      a.out_h[(int64_t)tok * a.ldo + mt * 8 + g] = __float2half_rn(silu_mul(lo, hi));
    } else {  // EPI_QKV: rows g and g+8 of the tile are the pair (i, i + d/2) of one head
      const int tiles_per_head = a.head_dim / 16, head = mt / tiles_per_head;
      const int ih = 8 * (mt - head * tiles_per_head) + g;
      const int row = head * a.head_dim + ih, row8 = row + a.head_dim / 2;
      __half* o = a.out_h + (int64_t)tok * a.ldo;
      __half y0, y1;
      if (head < a.n_rot_heads) {
        // round as the fp16 projection output, then rotate
        const float x0 = __half2float(__float2half_rn(lo)), x1 = __half2float(__float2half_rn(hi));
        const int pos = a.step->pos[tok], hd = a.head_dim / 2;
        const float cs = a.rope_cos[(int64_t)pos * hd + ih], sn = a.rope_sin[(int64_t)pos * hd + ih];
        y0 = __float2half_rn(x0 * cs - x1 * sn);
        y1 = __float2half_rn(x0 * sn + x1 * cs);
      } else {
        y0 = __float2half_rn(lo);
        y1 = __float2half_rn(hi);
      }
      o[row] = y0;
      o[row8] = y1;
      if (a.kv_store && head >= a.n_q_heads) {  // the token's own key (rotated) or value, into the FP16 pool
        const int Hkv = a.pool.n_kv_heads, which = head >= a.n_q_heads + Hkv ? 1 : 0;
        const int kvh = head - a.n_q_heads - which * Hkv, pos = a.step->pos[tok];
        const int blk = a.step->blk[tok];
        __half* v = reinterpret_cast<__half*>(pool_vec(a.pool, a.layer, blk, which, kvh, pos & 15));
        v[ih] = y0;
        v[ih + a.head_dim / 2] = y1;
      }
    }
  }
}

}  // namespace pipe
}  // namespace mag
