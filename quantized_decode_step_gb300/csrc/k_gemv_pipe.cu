// Decode GEMV for up to 4 tokens: one block per SM, a bulk-copy pipeline per warp.
//
// y[b][n] = sum_k deq(W)[n][k] x[b][k] ("5. Core modules" 5.1: 4-bit weights,
// FP16 activations; the 5.3 roofline makes this an HBM stream). Block i owns
// the contiguous 16-row tiles [T0, T1) of the matrix; a tile's 64-k chunks
// are contiguous in memory (640 bytes for W4, 2048 for fp16), so the block's
// weights are one contiguous run. The run is cut into one piece per warp
// (whole 4-chunk windows at batch 1); each warp streams its piece through its
// own ring of shared-memory slots with cp.async.bulk, one slot per copy,
// completing on the slot's mbarrier, and refills a slot as soon as it holds
// the slot in registers, so no warp ever waits on another to issue copies.
// The first two copies of every warp are issued before the wait on the
// previous kernel, whose outputs they do not touch, the rest once the
// activations are staged. A tile split between warps leaves each warp's partial in shared
// memory; the last warp to finish it adds the parts in warp order
// (deterministic) and runs the epilogue.
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
#include "pipe_dev.cuh"

namespace mag {

namespace {

using namespace pipe;


// WIN: batch 1, W4, K a multiple of 256 (the host checks): warps take whole 4-chunk windows (one ring
// slot each) and use the 8 MMA columns for the window's 8 groups rather than for tokens. Only that loop
// is compiled into such a kernel, which keeps its code (and instruction-cache footprint) small.
constexpr int kPreFills = 2;  // ring slots per warp filled before the wait on the previous kernel

template <int WFMT, int XSRC, int EPI, int B, bool WIN>
__device__ __forceinline__ void gemv_pipe_body(const GemvArgs& a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int CB = ChunkFmt<WFMT>::kBytes, SC = ChunkFmt<WFMT>::kPerSlot;
  constexpr uint32_t SB = SC * CB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int C = a.n_chunks, NS = a.stages;
  const int n_cta = gridDim.x, blk = blockIdx.x;
  // step timeline stamps (the tag is rebuilt from the arguments at each, so that nothing stays live)
  auto stamp = [&](unsigned int ev) {
    trace_stamp(a.trace, kTraceGemv | ((unsigned long long)a.n_mtiles << 32) | ((unsigned long long)a.n_chunks << 8) | B,
                ev);
  };
  if (tid == 0) stamp(0);
  const int T0 = (int)((int64_t)blk * a.n_mtiles / n_cta), T1 = (int)((int64_t)(blk + 1) * a.n_mtiles / n_cta);
  const int T = T1 - T0, P = T * C;  // the block's (tile, chunk) pairs, tile-major
  constexpr bool win = WIN;
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
    for (int f = 0; f < min(kPreFills, nf); ++f) issue(f);
  }
  for (int i = tid; i < a.t_max; i += kThreads) reinterpret_cast<uint32_t*>(smem + L.tcnt)[i] = 0;
  int* bounds = reinterpret_cast<int*>(smem + L.bounds);
  if (tid <= kCWarps) bounds[tid] = run_lo(tid);  // read after the staging's barriers
  __syncwarp();

  if (tid == 0) stamp(1);
  pdl_wait();
  pdl_trigger();
  const uint32_t xrow = C * 64 + 8, grow = 2 * C + 2;
  __half* xw = reinterpret_cast<__half*>(smem + L.x);
  float* xsw = reinterpret_cast<float*>(smem + L.xs);
  stage_x<WFMT, XSRC, B>(a, xw, xsw, reinterpret_cast<float*>(smem + L.red), xrow, grow, [] {});
  if (tid == 0) stamp(2);
  // the rest of the ring is filled once the activations are in: their loads must not queue behind it
  if (lane == 0)
    for (int f = kPreFills; f < min(NS, nf); ++f) issue(f);

  const uint4* xrow_l = reinterpret_cast<const uint4*>(xw + (size_t)min(g, B - 1) * xrow);
  const float2* X0p = reinterpret_cast<const float2*>(xsw + (size_t)min(2 * t, B - 1) * grow);
  const float2* X1p = reinterpret_cast<const float2*>(xsw + (size_t)min(2 * t + 1, B - 1) * grow);
  float4* part = reinterpret_cast<float4*>(smem + L.part);

  uint32_t* tcnt = reinterpret_cast<uint32_t*>(smem + L.tcnt);
  auto epilogue = [&](int tt, const float4 v) { tile_epilogue<EPI, B>(a, T0 + tt, v, g, t); };
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
  if constexpr (WIN) {
    // the current slot (as a pointer and as a 32-bit shared address) and its barrier
    const uint4* zero4 = reinterpret_cast<const uint4*>(smem + L.zero);
    const uint32_t ring_a = smem_u32(ring), bar0_a = smem_u32(full);
    uint32_t slot_a = ring_a, bar_a = bar0_a;
    const uint8_t* sp = ring;
    const uint8_t* nsrc = src + (int64_t)NS * SB;  // the fill that goes into the slot just read
    int nleft = n - NS * SC;                        // and its pairs
    for (int f = 0; f < nf; ++f) {
      if (!dead) {
        bool ok = mbar_try_wait_a(bar_a, round & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = mbar_wait_a(bar_a, round & 1, a.wait_limit);
          if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) atomicOr(a.err, 4u);
            dead = true;
          }
        }
      }
      uint4 w[SC], smq;
#pragma unroll
      for (int i = 0; i < SC; ++i) w[i] = *reinterpret_cast<const uint4*>(sp + i * CB + lane * 16);  // codes
      // (scale, min) of the window's groups 2t, 2t+1 (chunk t): rows g and g+8
      smq = *reinterpret_cast<const uint4*>(sp + t * CB + 512 + g * 16);
      __syncwarp();
      if (!dead && nleft > 0) {  // the slot is in registers: refill it (lane 0)
        bulk_copy_a(lane == 0, slot_a, nsrc, (uint32_t)min(SC, nleft) * CB, bar_a);
        ++issued;
      }
      nsrc += SB;
      nleft -= SC;
      const bool wrap = ++slot == NS;
      slot = wrap ? 0 : slot;
      round += wrap ? 1u : 0u;
      slot_a = wrap ? ring_a : slot_a + SB;
      bar_a = wrap ? bar0_a : bar_a + 8;
      sp = wrap ? ring : sp + SB;
      if (dead) continue;
      // column j of the MMAs = group j of the window: lane (g, t) feeds its activations only for j == g
      float d0[4], d1[4];
#pragma unroll
      for (int i = 0; i < SC; ++i)
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
          const uint4 xu = *(g == 2 * i + grp ? xrow_l + (c + i) * 8 + grp * 4 + t : zero4);
          const uint32_t wg = grp ? w[i].y : w[i].x, wv = grp ? w[i].w : w[i].z;
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
  } else {
  for (int f = 0; f < nf; ++f) {
    if (!dead) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(full + slot, round & 1, a.wait_limit));
      if (!ok) {
        if (lane == 0) atomicOr(a.err, 4u);
        dead = true;
      }
    }
    const int m = dead ? 0 : min(SC, n - f * SC);
    const uint8_t* sp = ring + (size_t)slot * SB;
    uint4 w[SC][2], wf[4];
    if (WFMT == W_W4) {
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
__global__ void __launch_bounds__(kThreads, 1) gemv_pipe_kernel(const GemvArgs a) {
  gemv_pipe_body<WFMT, XSRC, EPI, B, false>(a);
}

// The window kernels need no more than 80 registers a thread.
template <int WFMT, int XSRC, int EPI>
__global__ void __maxnreg__(80) gemv_win_kernel(const GemvArgs a) {
  gemv_pipe_body<WFMT, XSRC, EPI, 1, true>(a);
}

template <int WFMT, int XSRC, int EPI, int B, bool WIN>
cudaError_t launch_pipe_b(const Launch& L, const GemvArgs& a) {
  void (*kern)(const GemvArgs);
  if constexpr (WIN)
    kern = gemv_win_kernel<WFMT, XSRC, EPI>;
  else
    kern = gemv_pipe_kernel<WFMT, XSRC, EPI, B>;
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
    case 1:
      if (WFMT == W_W4 && a.n_chunks % 4 == 0) return launch_pipe_b<WFMT, XSRC, EPI, 1, WFMT == W_W4>(L, a);
      return launch_pipe_b<WFMT, XSRC, EPI, 1, false>(L, a);
    case 2: return launch_pipe_b<WFMT, XSRC, EPI, 2, false>(L, a);
    case 3: return launch_pipe_b<WFMT, XSRC, EPI, 3, false>(L, a);
    case 4: return launch_pipe_b<WFMT, XSRC, EPI, 4, false>(L, a);
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
