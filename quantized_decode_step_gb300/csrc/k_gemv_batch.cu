// W4A16 decode GEMV for 5 to 16 tokens: one block per SM, k-windows, bulk-copy rings per warp.
//
// y[b][n] = sum_k deq(W)[n][k] x[b][k] ("5. Core modules" 5.1: 4-bit weights,
// FP16 activations; by the 5.3 roofline the weights are still an HBM stream at
// 16 tokens: 16 multiply-adds per 0.625-byte weight). The grid is kw
// k-windows x tr tile ranges (kw x tr close to the SM count, one 512-thread
// block per SM). Block (range, window) stages the activations of its window
// once (16 tokens x 32 chunks of 64 k = 64 KB of fp16) and streams the
// window's part of its tiles: the block's slots (4 chunks of a tile, one
// 2,560-byte bulk copy) are cut into one contiguous run per warp, and each
// warp runs its own ring of slots completing on mbarriers, refilled as soon as
// the slot is in registers.
//
// Arithmetic per chunk (16 rows x 64 k) and 8-token column tile: the codes
// become fp16 subnormals by masks (pairs (k, k+4); the odd pairs' activations
// are staged divided by 16), two m16n8k16 MMAs per 32-group into a fresh
// accumulator, which the group's scale multiplies into the s-sum (units of
// 2^-24). The min terms sum_g m[n][g] X[b][g] (X = the group sums of the
// activations) are themselves a small product: per slot, two m16n8k8 MMAs of
// the 16 x 8 mins against X split into fp16 hi + lo (X - hi - lo below 2^-22 |X|).
// Nothing rounds the dequantised weights.
//
// A tile split between warps leaves each warp's part in shared memory, the last
// warp to leave its part adds them in warp order; a tile split between windows
// (kw > 1) leaves the block's sum in global memory and the last window to
// arrive (a per-tile counter) adds them in window order and runs the epilogue.
// Both orders are fixed, so the result does not depend on timing.
#include "kernels.h"
#include "gemv_epi.cuh"
#include "pipe_dev.cuh"

namespace mag {

namespace {

using pipe::bulk_copy;
using pipe::mbar_expect_tx;
using pipe::mbar_init;
using pipe::mbar_wait;
using pipe::mma_z;
using pipe::smem_u32;

constexpr int kWarps = 16, kThreads = kWarps * 32;
constexpr int kSlotChunks = 4;                             // chunks per ring slot
constexpr int kSlotBytes = kSlotChunks * kTileBytes;       // 2,560
constexpr int kMaxStages = 4;                              // ring slots per warp
constexpr int kPreFills = 2;                               // slots filled before the wait on the previous kernel
constexpr float kUnit = 16777216.0f;                       // 2^24: undoes the code scaling
static_assert(MAG_MAX_BATCH == 16, "the staging reads 16 partial sums of squares per tile");

// Dynamic shared memory of one block.
struct BatchSmem {
  uint32_t full, ring, x, xs, part, tcnt, bounds, red, total;
  uint32_t xrow, xsrow;  // halves per staged token row; uint2 per X row
};
__host__ __device__ inline BatchSmem batch_smem(int B, int NT, int cw, int stages, int t_max) {
  BatchSmem L;
  // +32 halves: rows g and g+1 of a quarter-warp's 16-byte loads sit 64 bytes apart in the banks
  L.xrow = (uint32_t)cw * 64 + 32;
  // one uint2 (X hi of the chunk's two groups, X lo of them) per chunk; rows 32 bytes apart mod 128
  L.xsrow = (uint32_t)cw + (uint32_t)(((4 - cw) % 16 + 16) % 16);
  L.full = 0;                                                // [warp][kMaxStages] mbarriers
  L.ring = kWarps * kMaxStages * 8;                          // [warp][stages][2,560]
  L.x = L.ring + (uint32_t)kWarps * stages * kSlotBytes;     // [B][xrow] fp16
  L.xs = L.x + (uint32_t)B * L.xrow * 2;                     // [B][xsrow] uint2
  L.part = L.xs + (uint32_t)B * L.xsrow * 8;                 // [warp][first / last tile][lane][NT] float4
  L.tcnt = L.part + (uint32_t)kWarps * 2 * 32 * NT * 16;     // per tile: warps done with their part
  L.bounds = L.tcnt + ((uint32_t)t_max * 4 + 15) / 16 * 16;  // first slot of every warp's run, and the end
  L.red = L.bounds + (kWarps + 1 + 3) / 4 * 16;              // [warp][16] partial sums, then 16 inverses
  L.total = L.red + (kWarps + 1) * MAG_MAX_BATCH * 4;
  return L;
}

// D += A(16x8, row) * B(8x8, col): a0 = A[g][2t..2t+1], a1 = A[g+8][2t..2t+1], b0 = B[2t..2t+1][g].
__device__ __forceinline__ void mma_1688(float* c, uint32_t a0, uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(b0));
}

// Stage chunks [c0, c1) of the B token rows: units of 8 activations in the order
// (x0,x4,x2,x6, x1/16,x5/16,x3/16,x7/16) (the MMAs' k order), and per chunk the fp16 hi / lo of its two group
// sums X (of the unscaled values). XSRC_RESID: x = fp16(r / sqrt(mean(r^2) + eps) * gamma), the mean from the
// producer's per-tile partial sums of squares.
template <int XSRC>
__device__ void stage_window(const GemvArgs& a, int c0, int c1, __half* xw, uint32_t xrow, __half* xsh,
                             uint32_t xsrow, float* red) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, B = a.batch;
  float* inv = red + kWarps * MAG_MAX_BATCH;
  if (XSRC == XSRC_RESID) {
    const int b = tid & 15;
    float s = 0.f;
    for (int i = tid >> 4; i < a.n_ss; i += kThreads / 16) s += __ldcg(a.ss_part + (int64_t)i * MAG_MAX_BATCH + b);
    s += __shfl_xor_sync(0xffffffffu, s, 16);
    if (lane < 16) red[warp * MAG_MAX_BATCH + lane] = s;
    __syncthreads();
    if (tid < B) {
      float tot = 0.f;
      for (int w = 0; w < kWarps; ++w) tot += red[w * MAG_MAX_BATCH + tid];
      inv[tid] = 1.0f / sqrtf(tot / (float)a.K + a.eps);
    }
    __syncthreads();
  }
  const int upr = (c1 - c0) * 8, U = B * upr;  // 8-value units per token row (a multiple of 4), in all
  constexpr int kAhead = 4;                    // units a thread loads before it converts them
  for (int base = 0; base < U; base += kAhead * kThreads) {
    float v[kAhead][8];
    uint4 h[kAhead];
#pragma unroll
    for (int q = 0; q < kAhead; ++q) {
      const int u = base + q * kThreads + tid;
      const int b = u / upr, k = (c0 * 8 + (u - b * upr)) * 8;
      const bool ok = u < U && k < a.K;
      if (XSRC == XSRC_RESID) {
        if (ok) {
          const float4 r0 = __ldcg(reinterpret_cast<const float4*>(a.r + (int64_t)b * a.ldr + k));
          const float4 r1 = __ldcg(reinterpret_cast<const float4*>(a.r + (int64_t)b * a.ldr + k + 4));
          v[q][0] = r0.x, v[q][1] = r0.y, v[q][2] = r0.z, v[q][3] = r0.w;
          v[q][4] = r1.x, v[q][5] = r1.y, v[q][6] = r1.z, v[q][7] = r1.w;
          h[q] = *reinterpret_cast<const uint4*>(a.gamma + k);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) v[q][e] = 0.f;
          h[q] = make_uint4(0, 0, 0, 0);
        }
      } else {
        // L2 only: the previous kernel wrote the activations
        h[q] = ok ? __ldcg(reinterpret_cast<const uint4*>(a.x + (int64_t)b * a.ldx + k)) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int q = 0; q < kAhead; ++q) {
      const int u = base + q * kThreads + tid;
      const bool live = u < U;
      const int b = live ? u / upr : 0, ul = live ? u - b * upr : 0;
      __half x8[8];
      if (XSRC == XSRC_RESID) {
        const float ib = live ? inv[b] : 0.f;
        const __half* gh = reinterpret_cast<const __half*>(&h[q]);
#pragma unroll
        for (int e = 0; e < 8; ++e) x8[e] = __float2half_rn(v[q][e] * ib * __half2float(gh[e]));
      } else {
        *reinterpret_cast<uint4*>(x8) = h[q];
      }
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) s += __half2float(x8[e]);
      if (live) {
        const __half k16 = __float2half_rn(0.0625f);
        __half o[8] = {x8[0], x8[4], x8[2], x8[6], __hmul(x8[1], k16), __hmul(x8[5], k16), __hmul(x8[3], k16),
                       __hmul(x8[7], k16)};
        *reinterpret_cast<uint4*>(xw + (size_t)b * xrow + 8 * ul) = *reinterpret_cast<const uint4*>(o);
      }
      // the 4 units of a 32-wide group are 4 consecutive lanes (u = tid mod 4 per unit, rows of whole groups)
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (live && (ul & 3) == 0) {
        const int gi = ul >> 2, cc = gi >> 1, grp = gi & 1;
        const __half hi = __float2half_rn(s), lo = __float2half_rn(s - __half2float(hi));
        __half* p = xsh + ((size_t)b * xsrow + cc) * 4;
        p[grp] = hi;
        p[2 + grp] = lo;
      }
    }
  }
  __syncthreads();
}

template <int NT, int XSRC, int EPI>
__global__ void __launch_bounds__(kThreads, 1) gemv_batch_kernel(const GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int B = a.batch, C = a.n_chunks, kw = a.ks, NS = a.stages;
  const int kwi = blockIdx.x % kw, tri = blockIdx.x / kw, tr = gridDim.x / kw;
  // step timeline stamps (the tag rebuilt from the arguments at each, so that nothing stays live)
  auto stamp = [&](unsigned int ev) {
    trace_stamp(a.trace, kTraceGemv | ((unsigned long long)a.n_mtiles << 32) | ((unsigned long long)a.n_chunks << 8) |
                             (unsigned)a.batch, ev);
  };
  if (tid == 0) stamp(0);
  const int T0 = (int)((int64_t)tri * a.n_mtiles / tr), T1 = (int)((int64_t)(tri + 1) * a.n_mtiles / tr);
  const int c0 = kwi * a.chunks_per_cta, c1 = min(C, c0 + a.chunks_per_cta);
  const int cb = c1 - c0, spt = (cb + kSlotChunks - 1) / kSlotChunks;  // chunks and slots per tile in the window
  const int S = (T1 - T0) * spt;                                        // the block's slots, tile-major
  auto run_lo = [&](int w) { return (int)((int64_t)S * w / kWarps); };  // first slot of warp w
  const int q0 = run_lo(warp), q1 = run_lo(warp + 1), nf = q1 - q0;
  const BatchSmem L = batch_smem(B, NT, a.chunks_per_cta, NS, a.t_max);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full) + warp * kMaxStages;
  uint8_t* ring = smem + L.ring + (size_t)warp * NS * kSlotBytes;
  // fill f: slot q0 + f of the block (chunks 4j .. 4j+3 of the window of tile T0 + ti) into ring slot f % NS
  auto issue = [&](int f) {
    const int s = q0 + f, ti = s / spt, j = s - ti * spt;
    const uint32_t bytes = (uint32_t)min(kSlotChunks, cb - kSlotChunks * j) * kTileBytes;
    uint64_t* bar = full + f % NS;
    mbar_expect_tx(bar, bytes);
    bulk_copy(ring + (size_t)(f % NS) * kSlotBytes,
              a.w + ((int64_t)(T0 + ti) * C + c0 + kSlotChunks * j) * kTileBytes, bytes, bar);
  };
  if (lane == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(full + i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the weights do not depend on earlier kernels: start streaming before waiting for them
    for (int f = 0; f < min(kPreFills, nf); ++f) issue(f);
  }
  uint32_t* tcnt = reinterpret_cast<uint32_t*>(smem + L.tcnt);
  for (int i = tid; i < a.t_max; i += kThreads) tcnt[i] = 0;
  int* bounds = reinterpret_cast<int*>(smem + L.bounds);
  if (tid <= kWarps) bounds[tid] = run_lo(tid);  // read after the staging's barrier
  __syncwarp();

  if (tid == 0) stamp(1);
  pdl_wait();
  pdl_trigger();
  __half* xw = reinterpret_cast<__half*>(smem + L.x);
  __half* xsh = reinterpret_cast<__half*>(smem + L.xs);
  stage_window<XSRC>(a, c0, c1, xw, L.xrow, xsh, L.xsrow, reinterpret_cast<float*>(smem + L.red));
  if (tid == 0) stamp(2);
  // the rest of the ring once the activations are in: their loads must not queue behind it
  if (lane == 0)
    for (int f = kPreFills; f < min(NS, nf); ++f) issue(f);

  // this lane's token rows (columns of the MMAs): g + 8 nt; past the batch, a valid row whose results are dropped
  const uint4* xr[NT];
  const uint2* xsr[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tok = min(g + 8 * nt, B - 1);
    xr[nt] = reinterpret_cast<const uint4*>(xw + (size_t)tok * L.xrow);
    xsr[nt] = reinterpret_cast<const uint2*>(xsh) + (size_t)tok * L.xsrow;
  }
  float4* part = reinterpret_cast<float4*>(smem + L.part);

  // a tile's window part is complete: with one window the epilogue runs at once; otherwise the part goes to
  // global memory and the last window to arrive adds the parts in window order
  auto window_done = [&](int ti, float (&r)[2][4]) {
    const int mt = T0 + ti;
    if (kw > 1) {
      float* p = a.partial + (((size_t)mt * kw + kwi) * 32 + lane) * (4 * NT);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        __stcg(reinterpret_cast<float4*>(p + 4 * nt), make_float4(r[nt][0], r[nt][1], r[nt][2], r[nt][3]));
      __threadfence();
      __syncwarp();
      uint32_t prev = 0;
      if (lane == 0) prev = atomicAdd(a.counters + mt, 1u);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if ((int)prev != kw - 1) return;
      __threadfence();
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) r[nt][j] = 0.f;
      for (int w = 0; w < kw; ++w) {
        const float* q = a.partial + (((size_t)mt * kw + w) * 32 + lane) * (4 * NT);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(q + 4 * nt));
          r[nt][0] += v.x, r[nt][1] += v.y, r[nt][2] += v.z, r[nt][3] += v.w;
        }
      }
      if (lane == 0) a.counters[mt] = 0;  // for the next launch (ordered by its wait on this grid)
    }
    tokepi::epilogue_tile<NT, EPI>(a, mt, r, lane);
  };
  auto overlaps = [&](int w, int tt) {
    const int a0 = bounds[w], a1 = bounds[w + 1];
    return a1 > a0 && a0 < (tt + 1) * spt && a1 > tt * spt;
  };
  // this warp's sums of tile ti: s-sums x 2^24 + min terms; a split tile's parts are added in warp order
  auto finish = [&](int ti, bool whole, int which, const float (&acc)[NT][8]) {
    float r[2][4] = {};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) r[nt][j] = fmaf(acc[nt][j], kUnit, acc[nt][4 + j]);
    if (whole) {
      window_done(ti, r);
      return;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      part[((warp * 2 + which) * 32 + lane) * NT + nt] = make_float4(r[nt][0], r[nt][1], r[nt][2], r[nt][3]);
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
    for (int w = 0; w < kWarps; ++w) n_parts += overlaps(w, ti);
    if ((int)prev + 1 < n_parts) return;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) r[nt][j] = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      if (!overlaps(w, ti)) continue;
      const int wh = ti == bounds[w] / spt ? 0 : 1;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float4 v = part[((w * 2 + wh) * 32 + lane) * NT + nt];
        r[nt][0] += v.x, r[nt][1] += v.y, r[nt][2] += v.z, r[nt][3] += v.w;
      }
    }
    window_done(ti, r);
  };

  bool dead = false;
  int ti = nf > 0 ? q0 / spt : 0, j = nf > 0 ? q0 - ti * spt : 0;
  const int t_first = ti;
  bool from_start = j == 0;  // this warp holds the current tile from the window's first slot
  float acc[NT][8];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[nt][i] = 0.f;
  int slot = 0;
  uint32_t round = 0;
  int issued = min(NS, nf);
  for (int f = 0; f < nf; ++f) {
    if (!dead && !__all_sync(0xffffffffu, mbar_wait(full + slot, round & 1, a.wait_limit))) {
      if (lane == 0) atomicOr(a.err, 4u);
      dead = true;
    }
    const int m = min(kSlotChunks, cb - kSlotChunks * j);  // chunks in this slot
    const uint8_t* sp = ring + (size_t)slot * kSlotBytes;
    uint4 cw[kSlotChunks], sm[kSlotChunks], smt = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < kSlotChunks; ++i)
      if (i < m) {
        cw[i] = *reinterpret_cast<const uint4*>(sp + i * kTileBytes + lane * 16);      // codes
        sm[i] = *reinterpret_cast<const uint4*>(sp + i * kTileBytes + 512 + g * 16);   // (scale, min)
      }
    if (t < m) smt = *reinterpret_cast<const uint4*>(sp + t * kTileBytes + 512 + g * 16);  // chunk t's mins
    __syncwarp();
    if (!dead && f + NS < nf) {  // the slot is in registers: refill it
      if (lane == 0) issue(f + NS);
      ++issued;
    }
    if (++slot == NS) {
      slot = 0;
      ++round;
    }
    if (!dead) {
#pragma unroll
      for (int i = 0; i < kSlotChunks; ++i) {
        if (i >= m) break;
        const int cc = kSlotChunks * j + i;  // chunk within the window
#pragma unroll
        for (int grp = 0; grp < 2; ++grp) {
          const uint32_t wg = grp ? cw[i].y : cw[i].x, wv = grp ? cw[i].w : cw[i].z;
          const uint32_t sg = wg >> 8, sv = wv >> 8;
          const float scg = __low2float(u32_as_h2(grp ? sm[i].y : sm[i].x));
          const float scv = __low2float(u32_as_h2(grp ? sm[i].w : sm[i].z));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint4 xu = xr[nt][cc * 8 + grp * 4 + t];
            float d[4];
            mma_z(d, wg & 0x000F000Fu, wv & 0x000F000Fu, sg & 0x000F000Fu, sv & 0x000F000Fu, xu.x, xu.y);
            mma_16816(d, wg & 0x00F000F0u, wv & 0x00F000F0u, sg & 0x00F000F0u, sv & 0x00F000F0u, xu.z, xu.w);
            acc[nt][0] = fmaf(scg, d[0], acc[nt][0]);
            acc[nt][1] = fmaf(scg, d[1], acc[nt][1]);
            acc[nt][2] = fmaf(scv, d[2], acc[nt][2]);
            acc[nt][3] = fmaf(scv, d[3], acc[nt][3]);
          }
        }
      }
      // min terms of the slot's 8 groups: A = mins [16 rows][8 groups], B = X [8 groups][8 tokens], hi and lo
      const uint32_t ma0 = __byte_perm(smt.x, smt.y, 0x7632), ma1 = __byte_perm(smt.z, smt.w, 0x7632);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint2 X = t < m ? xsr[nt][kSlotChunks * j + t] : make_uint2(0, 0);
        mma_1688(acc[nt] + 4, ma0, ma1, X.x);
        mma_1688(acc[nt] + 4, ma0, ma1, X.y);
      }
    }
    if (++j == spt) {  // end of the tile's window part
      finish(ti, from_start, 0, acc);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[nt][i] = 0.f;
      ++ti;
      j = 0;
      from_start = true;
    }
  }
  if (nf > 0 && j != 0) finish(ti, false, ti == t_first ? 0 : 1, acc);  // the run ends inside a tile
  if (dead && lane == 0) {
    // a wait gave up: do not leave with copies in flight (bounded waits for the last fill of every slot)
    for (int f = max(0, issued - NS); f < issued; ++f) mbar_wait(full + f % NS, (uint32_t)(f / NS) & 1);
  }
}

template <int NT, int XSRC, int EPI>
cudaError_t launch_nt(const Launch& Lc, const GemvArgs& a) {
  auto kern = gemv_batch_kernel<NT, XSRC, EPI>;
  const BatchSmem sl = batch_smem(a.batch, NT, a.chunks_per_cta, a.stages, a.t_max);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sl.total);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_cta * a.ks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sl.total;
  cfg.stream = Lc.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = Lc.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (Lc.counter) ++*Lc.counter;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int XSRC, int EPI>
cudaError_t launch_x(const Launch& L, const GemvArgs& a) {
  return a.batch > 8 ? launch_nt<2, XSRC, EPI>(L, a) : launch_nt<1, XSRC, EPI>(L, a);
}

}  // namespace

size_t gemv_batch_smem_bytes(int batch, int cw, int stages, int t_max) {
  return batch_smem(batch, batch > 8 ? 2 : 1, cw, stages, t_max).total;
}

int gemv_batch_max_stages() { return kMaxStages; }

size_t gemv_batch_stage_bytes() { return (size_t)kWarps * kSlotBytes; }

cudaError_t launch_gemv_batch(const Launch& L, const GemvArgs& a, int xsrc, int epi) {
  if (a.batch <= kPipeMaxBatch || a.batch > MAG_MAX_BATCH || a.stages < 2 || a.stages > kMaxStages ||
      a.n_cta < 1 || a.ks < 1 || a.chunks_per_cta < 1 || a.chunks_per_cta % kSlotChunks != 0 ||
      (int64_t)a.ks * a.chunks_per_cta < a.n_chunks || (int64_t)(a.ks - 1) * a.chunks_per_cta >= a.n_chunks ||
      a.n_cta > a.n_mtiles || a.t_max < (a.n_mtiles + a.n_cta - 1) / a.n_cta)
    return cudaErrorInvalidValue;
  if (xsrc == XSRC_RESID && epi == EPI_QKV) return launch_x<XSRC_RESID, EPI_QKV>(L, a);
  if (xsrc == XSRC_F16 && epi == EPI_RESID) return launch_x<XSRC_F16, EPI_RESID>(L, a);
  if (xsrc == XSRC_RESID && epi == EPI_SWIGLU) return launch_x<XSRC_RESID, EPI_SWIGLU>(L, a);
  return cudaErrorInvalidValue;
}

}  // namespace mag
