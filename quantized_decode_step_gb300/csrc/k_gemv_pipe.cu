// Decode GEMV for up to 4 tokens: one block per SM, a bulk-copy pipeline.
//
// y[b][n] = sum_k deq(W)[n][k] x[b][k] ("5. Core modules" 5.1: 4-bit weights,
// FP16 activations; the 5.3 roofline makes this an HBM stream). Block i owns
// the contiguous 16-row tiles [T0, T1) of the matrix; a tile's 64-k chunks
// are contiguous in memory (640 bytes for W4, 2048 for fp16), so the block's
// weights are one contiguous run, streamed into a ring of shared-memory
// stages with cp.async.bulk, one stage (up to 16 chunks of one tile) per
// copy, completing on the stage's mbarrier; the first copies are issued
// before the wait on the previous kernel, whose outputs they do not touch.
// The 16 warps take chunk c of every stage with c mod 16 = warp and release
// the stage once the chunk is in registers; the last warp to release a stage
// refills it with the stage S ahead (a shared-memory counter per slot, so no
// warp ever waits for another to issue copies). Each warp accumulates a
// partial of the tile; at the tile's end the partials meet in shared memory
// and the tile's owner warp adds them in warp order (deterministic). The
// epilogue runs once for the whole block.
//
// W4 arithmetic: each 32-bit word of codes holds the k-values 8t..8t+7 of a
// row. Masking it (and the word shifted right by 8) with 0x000F000F and
// 0x00F000F0 leaves pairs of codes in the mantissa of two fp16 subnormals:
// (k0,k4) and (k2,k6) as code * 2^-24, (k1,k5) and (k3,k7) as code * 2^-20.
// The activations of the second kind are staged divided by 16 (exact for
// |x| >= 2^-10; below that the change is under 2^-25), so both m16n8k16 MMAs
// of a 32-wide group accumulate code * x in units of 2^-24 without any
// rounding of the dequantised weights, and per group
//     sum_k (s q_k + m) x_k = s * 2^24 * acc + m * X_g,   X_g = sum_k x_k.
// The pre-norm RMSNorm of the QKV, gate-up and LM-head inputs is computed by
// every block from the fp32 residual while staging.
#include "kernels.h"

namespace mag {

namespace {

constexpr int kCWarps = 16;                     // warps per block
constexpr int kThreads = kCWarps * 32;
constexpr int kMaxSlots = 8;                    // ring slots per warp
constexpr uint32_t kSpinLimit = 1u << 22;       // mbarrier polls before a wait is declared stuck
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
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(b, parity)) return true;
  return false;
}
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
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
      h = ok ? *reinterpret_cast<const uint4*>(a.x + (int64_t)b * a.ldx + k) : make_uint4(0, 0, 0, 0);
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

template <int WFMT, int XSRC, int EPI, int B>
__global__ void __launch_bounds__(kThreads, 1) gemv_pipe_kernel(const GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int CB = ChunkFmt<WFMT>::kBytes, SC = ChunkFmt<WFMT>::kPerSlot;
  constexpr uint32_t SB = SC * CB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int C = a.n_chunks, NS = a.stages;
  const int n_cta = gridDim.x, blk = blockIdx.x;
  const int T0 = (int)((int64_t)blk * a.n_mtiles / n_cta), T1 = (int)((int64_t)(blk + 1) * a.n_mtiles / n_cta);
  const int T = T1 - T0, P = T * C;  // the block's (tile, chunk) pairs, tile-major
  // Batch 1, W4, K a multiple of 256: warps take whole 4-chunk windows (one ring slot each) and use
  // the 8 MMA columns for the window's 8 groups rather than for tokens.
  const bool win = WFMT == W_W4 && B == 1 && C % 4 == 0;
  const int U = win ? 4 : 1;
  auto run_lo = [&](int w) { return U * (int)((int64_t)(P / U) * w / kCWarps); };  // first pair of warp w
  const int q0 = run_lo(warp), q1 = run_lo(warp + 1);
  const int n = q1 - q0, nf = (n + SC - 1) / SC;  // this warp's pairs and ring fills
  const PipeSmem L = pipe_smem(WFMT, B, C, NS, a.t_max);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full) + warp * kMaxSlots;
  uint8_t* ring = smem + L.ring + (size_t)warp * NS * SB;
  const uint8_t* src = a.w + ((int64_t)T0 * C + q0) * CB;
  // fill f: pairs [q0 + f SC, + SC) of this warp into slot f % NS, one bulk copy
  auto issue = [&](int f) {
    const uint32_t bytes = (uint32_t)min(SC, n - f * SC) * CB;
    uint64_t* bar = full + f % NS;
    mbar_expect_tx(bar, bytes);
    bulk_copy(ring + (size_t)(f % NS) * SB, src + (int64_t)f * SB, bytes, bar);
  };
  if (tid == 0) *reinterpret_cast<uint4*>(smem + L.zero) = make_uint4(0, 0, 0, 0);
  if (lane == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(full + i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the weights do not depend on earlier kernels: start streaming before waiting for them
    for (int f = 0; f < min(NS, nf); ++f) issue(f);
  }
  for (int i = tid; i < a.t_max; i += kThreads) reinterpret_cast<uint32_t*>(smem + L.tcnt)[i] = 0;
  int* bounds = reinterpret_cast<int*>(smem + L.bounds);
  if (tid <= kCWarps) bounds[tid] = run_lo(tid);  // read after the staging's barriers
  __syncwarp();

  pdl_wait();
  pdl_trigger();
  const uint32_t xrow = C * 64 + 8, grow = 2 * C + 2;
  __half* xw = reinterpret_cast<__half*>(smem + L.x);
  float* xsw = reinterpret_cast<float*>(smem + L.xs);
  stage_x<WFMT, XSRC, B>(a, xw, xsw, reinterpret_cast<float*>(smem + L.red), xrow, grow, [] {});

  const uint4* xrow_l = reinterpret_cast<const uint4*>(xw + (size_t)min(g, B - 1) * xrow);
  const float2* X0p = reinterpret_cast<const float2*>(xsw + (size_t)min(2 * t, B - 1) * grow);
  const float2* X1p = reinterpret_cast<const float2*>(xsw + (size_t)min(2 * t + 1, B - 1) * grow);
  float4* part = reinterpret_cast<float4*>(smem + L.part);

  uint32_t* tcnt = reinterpret_cast<uint32_t*>(smem + L.tcnt);
  // v: (row g, token 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1) of tile tt
  auto epilogue = [&](int tt, const float4 v) {
    const int mt = T0 + tt;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int tok = 2 * t + jj;
      if (tok >= B) continue;
      const float lo = jj ? v.y : v.x, hi = jj ? v.w : v.z;  // rows g and g + 8 of the tile
      if (EPI == EPI_RESID) {
        float* o = a.r + (int64_t)tok * a.ldr + mt * 16 + g;
        o[0] += lo;
        o[8] += hi;
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
        if (head < a.n_rot_heads) {
          // round as the fp16 projection output, then rotate
          const float x0 = __half2float(__float2half_rn(lo)), x1 = __half2float(__float2half_rn(hi));
          const int pos = a.step->pos[tok], hd = a.head_dim / 2;
          const float cs = a.rope_cos[(int64_t)pos * hd + ih], sn = a.rope_sin[(int64_t)pos * hd + ih];
          o[row] = __float2half_rn(x0 * cs - x1 * sn);
          o[row8] = __float2half_rn(x0 * sn + x1 * cs);
        } else {
          o[row] = __float2half_rn(lo);
          o[row8] = __float2half_rn(hi);
        }
      }
    }
  };
  auto overlaps = [&](int w, int tt) {
    const int a0 = bounds[w], a1 = bounds[w + 1];
    return a1 > a0 && a0 < (tt + 1) * C && a1 > tt * C;
  };
  // a finished tile: a whole one goes straight to the epilogue; a split one leaves this warp's part, and
  // the last warp to leave its part adds them all in warp order (deterministic) and runs the epilogue
  auto finish = [&](int ti, bool whole, int which, const float (&acc)[8]) {
    float4 r4;
    if (WFMT == W_W4) {
      r4 = make_float4(fmaf(acc[0], kCodeUnit, acc[4]), fmaf(acc[1], kCodeUnit, acc[5]),
                       fmaf(acc[2], kCodeUnit, acc[6]), fmaf(acc[3], kCodeUnit, acc[7]));
    } else {
      r4 = make_float4(acc[0], acc[1], acc[2], acc[3]);
    }
    if (whole) {
      epilogue(ti, r4);
      return;
    }
    part[(warp * 2 + which) * 32 + lane] = r4;
    __syncwarp();
    uint32_t prev = 0;
    if (lane == 0)
      asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                   : "=r"(prev)
                   : "r"(smem_u32(tcnt + ti))
                   : "memory");
    prev = __shfl_sync(0xffffffffu, prev, 0);
    __syncwarp();
    int n_parts = 0;
    for (int w = 0; w < kCWarps; ++w) n_parts += overlaps(w, ti);
    if ((int)prev + 1 < n_parts) return;
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int w = 0; w < kCWarps; ++w) {
      if (!overlaps(w, ti)) continue;
      const float4 v = part[(w * 2 + (ti == bounds[w] / C ? 0 : 1)) * 32 + lane];
      sum.x += v.x, sum.y += v.y, sum.z += v.z, sum.w += v.w;
    }
    epilogue(ti, sum);
  };

  // window path: a lane holds the sums of its own groups; the row totals are the sums over the quad
  auto quad_sum = [&](const float (&v)[8], float (&o)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float x = v[j];
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      o[j] = x;
    }
  };

  bool dead = false;
  int ti = n > 0 ? q0 / C : 0, c = n > 0 ? q0 - ti * C : 0;
  const int t_first = ti;
  bool from_start = c == 0;  // this warp holds the current tile from its chunk 0
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int slot = 0;
  uint32_t round = 0;
  int issued = min(NS, nf);  // fills issued so far
  for (int f = 0; f < nf; ++f) {
    if (!dead) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(full + slot, round & 1));
      if (!ok) {
        if (lane == 0) atomicOr(a.err, 4u);
        dead = true;
      }
    }
    const int m = dead ? 0 : min(SC, n - f * SC);
    const uint8_t* sp = ring + (size_t)slot * SB;
    uint4 w[SC][2], wf[4], smq;
    if (WFMT == W_W4 && win) {
#pragma unroll
      for (int i = 0; i < SC; ++i)
        if (i < m) w[i][0] = *reinterpret_cast<const uint4*>(sp + i * CB + lane * 16);  // codes
      // (scale, min) of the window's groups 2t, 2t+1 (chunk t): rows g and g+8
      if (m > 0) smq = *reinterpret_cast<const uint4*>(sp + t * CB + 512 + g * 16);
    } else if (WFMT == W_W4) {
#pragma unroll
      for (int i = 0; i < SC; ++i)
        if (i < m) {
          w[i][0] = *reinterpret_cast<const uint4*>(sp + i * CB + lane * 16);      // codes
          w[i][1] = *reinterpret_cast<const uint4*>(sp + i * CB + 512 + g * 16);   // (scale, min)
        }
    } else if (m > 0) {
      const uint4* p4 = reinterpret_cast<const uint4*>(sp + lane * 64);
      wf[0] = p4[0], wf[1] = p4[1], wf[2] = p4[2], wf[3] = p4[3];
    }
    __syncwarp();
    if (!dead && f + NS < nf) {  // the slot is in registers: refill it
      if (lane == 0) issue(f + NS);
      ++issued;
    }
    if (++slot == NS) {
      slot = 0;
      ++round;
    }
    if (WFMT == W_W4 && B == 1 && win) {
      if (m == SC) {
        // column j of the MMAs = group j of the window: lane (g, t) feeds its activations only for j == g
        const uint4* zero4 = reinterpret_cast<const uint4*>(smem + L.zero);
        float d0[4], d1[4];
#pragma unroll
        for (int i = 0; i < SC; ++i)
#pragma unroll
          for (int grp = 0; grp < 2; ++grp) {
            const uint4 xu = *(g == 2 * i + grp ? xrow_l + (c + i) * 8 + grp * 4 + t : zero4);
            const uint32_t wg = grp ? w[i][0].y : w[i][0].x, wv = grp ? w[i][0].w : w[i][0].z;
            const uint32_t sg = wg >> 8, sv = wv >> 8;
            float* d = (i & 1) ? d1 : d0;
            if (i < 2 && grp == 0)
              mma_z(*reinterpret_cast<float(*)[4]>(d), wg & 0x000F000Fu, wv & 0x000F000Fu, sg & 0x000F000Fu,
                    sv & 0x000F000Fu, xu.x, xu.y);
            else
              mma_16816(d, wg & 0x000F000Fu, wv & 0x000F000Fu, sg & 0x000F000Fu, sv & 0x000F000Fu, xu.x, xu.y);
            mma_16816(d, wg & 0x00F000F0u, wv & 0x00F000F0u, sg & 0x00F000F0u, sv & 0x00F000F0u, xu.z, xu.w);
          }
        // d: (row g, group 2t), (row g, 2t+1), (row g+8, 2t), (row g+8, 2t+1), in units of 2^-24
        const float2 X = X0p[c + t];
        const float2 f0 = __half22float2(u32_as_h2(smq.x)), f1 = __half22float2(u32_as_h2(smq.y));
        const float2 f2 = __half22float2(u32_as_h2(smq.z)), f3 = __half22float2(u32_as_h2(smq.w));
        acc[0] = fmaf(f0.x, d0[0] + d1[0], fmaf(f1.x, d0[1] + d1[1], acc[0]));
        acc[2] = fmaf(f2.x, d0[2] + d1[2], fmaf(f3.x, d0[3] + d1[3], acc[2]));
        acc[4] = fmaf(f0.y, X.x, fmaf(f1.y, X.y, acc[4]));
        acc[6] = fmaf(f2.y, X.x, fmaf(f3.y, X.y, acc[6]));
        c += SC;
        if (c == C) {  // end of a tile
          float q[8];
          quad_sum(acc, q);
          finish(ti, from_start, 0, q);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] = 0.f;
          ++ti;
          c = 0;
          from_start = true;
        }
      }
      continue;
    }
#pragma unroll
    for (int i = 0; i < SC; ++i) {
      if (i >= m) break;
      if (WFMT == W_W4) {
        const uint4 xa = xrow_l[c * 8 + t], xb = xrow_l[c * 8 + 4 + t];
        const float2 X0 = X0p[c], X1 = B > 1 ? X1p[c] : X0;
        w4_chunk<B>(w[i][0], w[i][1], xa, xb, X0, X1, acc);
      } else {
        // rows g (wf[0], wf[1]) and g+8 (wf[2], wf[3]) at k = 64c + 16t .. +15, natural activation order
        const uint4 x0 = xrow_l[c * 8 + 2 * t], x1 = xrow_l[c * 8 + 2 * t + 1];
        mma_16816(acc, wf[0].x, wf[2].x, wf[0].y, wf[2].y, x0.x, x0.y);
        mma_16816(acc, wf[0].z, wf[2].z, wf[0].w, wf[2].w, x0.z, x0.w);
        mma_16816(acc, wf[1].x, wf[3].x, wf[1].y, wf[3].y, x1.x, x1.y);
        mma_16816(acc, wf[1].z, wf[3].z, wf[1].w, wf[3].w, x1.z, x1.w);
      }
      if (++c == C) {  // end of a tile
        finish(ti, from_start, 0, acc);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
        ++ti;
        c = 0;
        from_start = true;
      }
    }
  }
  if (n > 0 && c != 0) {  // the run ends inside a tile
    float q[8];
    if (win) quad_sum(acc, q);
    finish(ti, false, ti == t_first ? 0 : 1, win ? q : acc);
  }
  if (dead && lane == 0) {
    // a wait gave up: do not leave with copies in flight (bounded waits for the last fill of every slot)
    for (int f = max(0, issued - NS); f < issued; ++f) mbar_wait(full + f % NS, (uint32_t)(f / NS) & 1);
  }
}

template <int WFMT, int XSRC, int EPI, int B>
cudaError_t launch_pipe_b(const Launch& L, const GemvArgs& a) {
  auto kern = gemv_pipe_kernel<WFMT, XSRC, EPI, B>;
  const PipeSmem sl = pipe_smem(WFMT, B, a.n_chunks, a.stages, a.t_max);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sl.total);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_cta);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sl.total;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.counter) ++*L.counter;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int WFMT, int XSRC, int EPI>
cudaError_t launch_pipe_t(const Launch& L, const GemvArgs& a) {
  switch (a.batch) {
    case 1: return launch_pipe_b<WFMT, XSRC, EPI, 1>(L, a);
    case 2: return launch_pipe_b<WFMT, XSRC, EPI, 2>(L, a);
    case 3: return launch_pipe_b<WFMT, XSRC, EPI, 3>(L, a);
    case 4: return launch_pipe_b<WFMT, XSRC, EPI, 4>(L, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t gemv_pipe_smem_bytes(int wfmt, int batch, int n_chunks, int stages, int t_max) {
  return pipe_smem(wfmt, batch, n_chunks, stages, t_max).total;
}

int gemv_pipe_max_stages() { return kMaxSlots; }

size_t gemv_pipe_slot_bytes(int wfmt) { return (size_t)kCWarps * slot_bytes(wfmt); }

cudaError_t launch_gemv_pipe(const Launch& L, const GemvArgs& a, int wfmt, int xsrc, int epi) {
  if (a.batch < 1 || a.batch > kPipeMaxBatch || a.stages < 2 || a.stages > kMaxSlots || a.n_cta < 1)
    return cudaErrorInvalidValue;
#define MAG_PIPE_CASE(W_, X_, E_) \
  if (wfmt == W_ && xsrc == X_ && epi == E_) return launch_pipe_t<W_, X_, E_>(L, a);
  MAG_PIPE_CASE(W_W4, XSRC_RESID, EPI_QKV)
  MAG_PIPE_CASE(W_W4, XSRC_F16, EPI_RESID)
  MAG_PIPE_CASE(W_W4, XSRC_RESID, EPI_SWIGLU)
  MAG_PIPE_CASE(W_F16, XSRC_RESID, EPI_STORE_OUT)
#undef MAG_PIPE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace mag
