// Chunked prefill: the dense contractions of a T-token chunk on the 5th-generation
// tensor cores (tcgen05 MMA, accumulator in tensor memory, operands staged by TMA),
// plus the row-wise pieces around them.
//
// The chunk's projections are GEMMs Y[T][N] = X[T][K] W[N][K]^T. The W4 weights
// can not be expanded inside the GEMM at tensor-core speed (at ~1 PFLOP/s an SM
// has well under one ALU instruction per weight and token-tile), and rounding the
// dequantised value s q + m to fp16 alone leaves an error that 32 layers amplify
// beyond the tolerance. So at load time every projection also gets an exact
// two-term fp16 copy, w = hi + lo (hi = fp16(w), lo = fp16(w - hi); w = s q + m
// is exact in fp32), and the GEMM accumulates X hi^T + X lo^T in one fp32
// accumulator: twice the tensor work, no rounding of the weights.
//
// GEMM block (persistent, one per SM): 128 x 128 output tiles, K in steps of 64.
// Warp 0 issues the TMA loads (A, hi, lo; 128-byte swizzle) into a 4-stage ring;
// one thread of warp 1 issues tcgen05.mma (M 128, N 128, K 16; fp16 in, fp32 out
// in one of two 128-column TMEM accumulators) and commits each stage back to the
// producer; warps 2-5 read the accumulator with tcgen05.ld (each warp its 32 TMEM
// lanes = 32 rows) and apply the epilogue while the next tile accumulates.
#include <cuda.h>

#include <algorithm>

#include "kernels.h"

namespace mag {

namespace {

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4;
constexpr int TILE_A = BM * BK * 2, TILE_B = BN * BK * 2;
constexpr int STAGE_BYTES = TILE_A + 2 * TILE_B;
constexpr int kGemmThreads = 192;
constexpr uint32_t kSpin = 1u << 24;

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void mb_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mb_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t* b, uint32_t par) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(par)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mb_wait(uint64_t* b, uint32_t par) {
  for (uint32_t i = 0; i < kSpin; ++i)
    if (mb_try(b, par)) return true;
  return false;
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(su32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}
// Shared-memory matrix descriptor: K-major rows of 128 bytes, 128-byte swizzle,
// 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(const void* p) {
  uint64_t d = (static_cast<uint64_t>(su32(p)) & 0x3FFFFull) >> 4;
  d |= 1ull << 16;            // leading-dimension offset (not used by this layout)
  d |= (1024ull >> 4) << 32;  // stride-dimension offset
  d |= 1ull << 46;            // descriptor version
  d |= 2ull << 61;            // 128-byte swizzle
  return d;
}
// Instruction descriptor of kind::f16: fp16 A and B (K-major), fp32 D, M 128, N 128.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}
// 32 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ float silu_mul(float gte, float up) { return gte / (1.0f + expf(-gte)) * up; }

constexpr int kSq = 36;                              // floats per staged row (see the epilogue)
constexpr int kStageSqBytes = 32 * kSq * 4;          // one warp's 32 x 32 staging square
constexpr int kGemmSmem = STAGES * STAGE_BYTES + 4 * kStageSqBytes + 256 + 1024;

// Persistent: one block per SM takes output tiles tile = blockIdx.x + i gridDim.x, the token tiles of a
// weight tile next to each other (they run at the same time and share its bytes through L2). The ring
// of stages runs on across tiles, and the accumulator is double-buffered in tensor memory, so the
// epilogue of tile i overlaps the MMAs of tile i + 1.
template <int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_hi,
                   const __grid_constant__ CUtensorMap map_lo, const TcGemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* stage_sq = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + 4 * kStageSqBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;   // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_m = (a.M + BM - 1) / BM, n_tiles = n_m * (a.N / BN);
  const int nk = (a.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mb_init(full + s, 1);
      mb_init(empty + s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mb_init(acc_full + i, 1);
      mb_init(acc_empty + i, 4);  // one arrival per epilogue warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "n"(2 * BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer: the first tile's first stages of weights before waiting for the previous kernel
    // (they do not depend on it), then everything in ring order
    if (lane == 0 && (int)blockIdx.x < n_tiles) {
      const int pre = min(STAGES, nk);
      {
        const int n0 = ((int)blockIdx.x / n_m) * BN;
        for (int kb = 0; kb < pre; ++kb) {
          uint8_t* st = smem + kb * STAGE_BYTES;
          mb_expect(full + kb, STAGE_BYTES);
          tma_2d(st + TILE_A, &map_hi, kb * BK, n0, full + kb);
          tma_2d(st + TILE_A + TILE_B, &map_lo, kb * BK, n0, full + kb);
        }
        pdl_wait();
        const int m0 = ((int)blockIdx.x % n_m) * BM;
        for (int kb = 0; kb < pre; ++kb) tma_2d(smem + kb * STAGE_BYTES, &map_a, kb * BK, m0, full + kb);
      }
      int g = 0;  // stages issued so far, over all tiles
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int m0 = (tile % n_m) * BM, n0 = (tile / n_m) * BN;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          if (g < pre) continue;  // issued above
          const int s = g % STAGES;
          if (!mb_wait(empty + s, ((g / STAGES) - 1) & 1)) {
            atomicOr(a.err, 8u);
            ok = false;
            break;
          }
          uint8_t* st = smem + s * STAGE_BYTES;
          mb_expect(full + s, STAGE_BYTES);
          tma_2d(st + TILE_A, &map_hi, kb * BK, n0, full + s);
          tma_2d(st + TILE_A + TILE_B, &map_lo, kb * BK, n0, full + s);
          tma_2d(st, &map_a, kb * BK, m0, full + s);
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: tile i into accumulator buffer i % 2, once the epilogue has drained it
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int tile = blockIdx.x, it = 0; tile < n_tiles && ok; tile += gridDim.x, ++it) {
        const int ab = it & 1;
        if (it >= 2 && !mb_wait(acc_empty + ab, ((it >> 1) - 1) & 1)) {
          atomicOr(a.err, 64u);
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d = tmem + (uint32_t)(ab * BN);
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % STAGES;
          if (!mb_wait(full + s, (g / STAGES) & 1)) {
            atomicOr(a.err, 16u);
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          uint8_t* st = smem + s * STAGE_BYTES;
          const uint64_t da = smem_desc(st), dh = smem_desc(st + TILE_A), dl = smem_desc(st + TILE_A + TILE_B);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t off = (uint64_t)(k * 32) >> 4;  // 16 fp16 further along K
            mma_f16(d, da + off, dh + off, (kb | k) != 0);
            mma_f16(d, da + off, dl + off, 1);
          }
          mma_commit(empty + s);
        }
        if (ok) mma_commit(acc_full + ab);
      }
    }
  } else {
    // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 = rows of the tile. A thread holds one row;
    // the warp passes each 32-column slice through its own padded shared-memory square so that global
    // memory sees whole 16-byte runs of a row.
    pdl_wait();
    pdl_trigger();
    const int q = warp & 3;
    float* sq = stage_sq + q * 32 * kSq;
    // this lane's row of the square <- v (32 values); float4 stores of a quarter-warp on distinct banks
    auto put_row = [&](const float (&v)[32]) {
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(sq + lane * kSq + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    };
    // row rr, columns 4 c4 .. 4 c4 + 3 of the square
    auto get4 = [&](int rr, int c4) { return *reinterpret_cast<const float4*>(sq + rr * kSq + 4 * c4); };
    // the square's 32 rows x 32 columns as fp16 at out (row stride ldo), rows from row0, valid rows < M
    auto store_f16 = [&](__half* out, int row0, int ld, bool col_ok) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = (lane >> 2) + 8 * i, c8 = lane & 3;
        if (row0 + rr < a.M && col_ok) {
          const float4 y0 = get4(rr, 2 * c8), y1 = get4(rr, 2 * c8 + 1);
          uint4 h;
          h.x = h2_as_u32(__floats2half2_rn(y0.x, y0.y));
          h.y = h2_as_u32(__floats2half2_rn(y0.z, y0.w));
          h.z = h2_as_u32(__floats2half2_rn(y1.x, y1.y));
          h.w = h2_as_u32(__floats2half2_rn(y1.z, y1.w));
          *reinterpret_cast<uint4*>(out + (int64_t)(row0 + rr) * ld + 8 * c8) = h;
        }
      }
    };
    for (int tile = blockIdx.x, it = 0; tile < n_tiles; tile += gridDim.x, ++it) {
      const int ab = it & 1;
      const int m0 = (tile % n_m) * BM, n0 = (tile / n_m) * BN;
      const int m = m0 + q * 32 + lane, row0 = m0 + q * 32;
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * BN);
      if (!mb_wait(acc_full + ab, (it >> 1) & 1)) {
        atomicOr(a.err, 32u);
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (EPI == EPI_RESID) {
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          tmem_ld32(trow + c0, v);
          put_row(v);
          __syncwarp();
          // 32 rows x 8 float4: lane takes float4 (lane & 7) of rows lane / 8 + 4 i; all loads first
          const int c4 = lane & 7, col = n0 + c0 + 4 * c4;
          float4 y[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = (lane >> 3) + 4 * i;
            y[i] = (row0 + rr < a.M && col < a.n_valid)
                       ? *reinterpret_cast<const float4*>(a.r + (int64_t)(row0 + rr) * a.ldr + col)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = (lane >> 3) + 4 * i;
            if (row0 + rr < a.M && col < a.n_valid) {
              const float4 x = get4(rr, c4);
              *reinterpret_cast<float4*>(a.r + (int64_t)(row0 + rr) * a.ldr + col) =
                  make_float4(y[i].x + x.x, y[i].y + x.y, y[i].z + x.z, y[i].w + x.w);
            }
          }
          __syncwarp();
        }
      } else if (EPI == EPI_SWIGLU) {
        // tile columns [0, 64) are gate rows 64 (n0/128) + c, [64, 128) the matching up rows
        for (int c0 = 0; c0 < BN / 2; c0 += 32) {
          float g[32], u[32];
          tmem_ld32(trow + c0, g);
          tmem_ld32(trow + c0 + BN / 2, u);
#pragma unroll
          for (int j = 0; j < 32; ++j) g[j] = silu_mul(g[j], u[j]);
          put_row(g);
          __syncwarp();
          const int j0 = (n0 / BN) * (BN / 2) + c0;
          store_f16(a.out + j0, row0, a.ldo, j0 + 8 * (lane & 3) < a.n_valid);
          __syncwarp();
        }
      } else {  // EPI_QKV: fp16 q, k, v; q and k rotated at position pos0 + m (pairs (i, i + d/2) of a head)
        const int d = a.head_dim, hd = d / 2;
        const int mm = min(m, a.M - 1);  // rows past the chunk compute, but store nothing
        const int pos = a.row_pos ? a.row_pos[mm] : a.pos0 + mm;
        for (int c0 = 0; c0 < BN; c0 += 32) {
          const int head = (n0 + c0) / d, i0 = (n0 + c0) - head * d;
          if (i0 >= hd) continue;  // the second half of a head comes with the first
          float x0[32], x1[32];
          tmem_ld32(trow + c0, x0);
          tmem_ld32(trow + c0 + hd, x1);
          if (head < a.n_rot_heads) {
            const float4* cs = reinterpret_cast<const float4*>(a.rope_cos + (int64_t)pos * hd + i0);
            const float4* sn = reinterpret_cast<const float4*>(a.rope_sin + (int64_t)pos * hd + i0);
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 c = cs[j4], sv = sn[j4];
              const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                // round as the fp16 projection output, then rotate
                const int j = 4 * j4 + e;
                const float a0 = __half2float(__float2half_rn(x0[j])), a1 = __half2float(__float2half_rn(x1[j]));
                x0[j] = a0 * cc[e] - a1 * ss[e];
                x1[j] = a0 * ss[e] + a1 * cc[e];
              }
            }
          }
          put_row(x0);
          __syncwarp();
          store_f16(a.out + n0 + c0, row0, a.ldo, true);
          __syncwarp();
          put_row(x1);
          __syncwarp();
          store_f16(a.out + n0 + c0 + hd, row0, a.ldo, true);
          __syncwarp();
        }
      }
      // the accumulator buffer is drained: the MMA warp may reuse it
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(acc_empty + ab)) : "memory");
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(2 * BN) : "memory");
}

// ---------------------------------------------------------------- row kernels
// One block per token row: r = fp32(x).
__global__ void rows_to_resid_kernel(const __half* __restrict__ x, float* __restrict__ r, int D) {
  const int64_t row = blockIdx.x;
  for (int i = threadIdx.x; i < D; i += blockDim.x) r[row * D + i] = __half2float(x[row * D + i]);
}

// One block per listed row: dst row i = src row rows.row[i] (the last rows of several sessions' chunks).
__global__ void gather_rows_kernel(const float* __restrict__ src, int D, const RowList rows, float* __restrict__ dst) {
  pdl_wait();
  pdl_trigger();
  const int64_t from = rows.row[blockIdx.x];
  for (int i = threadIdx.x; i < D; i += blockDim.x) dst[(int64_t)blockIdx.x * D + i] = src[from * D + i];
}

// One block per token row: xn = fp16(r / sqrt(mean(r^2) + eps) * gamma) ("5. Core modules" 5.1, pre-norm).
// D % 4 == 0: each thread keeps its float4 units of the row in registers (one pass over memory) when the
// row fits kRegUnits units a thread, else reads them twice.
constexpr int kNormThreads = 256, kRegUnits = 8;
__global__ void __launch_bounds__(kNormThreads) rmsnorm_rows_kernel(const float* __restrict__ r,
                                                                    const __half* __restrict__ gamma, float eps,
                                                                    int D, __half* __restrict__ xn) {
  __shared__ float red[kNormThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int64_t row = blockIdx.x;
  const float4* rr = reinterpret_cast<const float4*>(r + row * D);
  const int U = D / 4;
  const bool in_regs = U <= kRegUnits * kNormThreads;
  float4 v[kRegUnits];
  float ss = 0.f;
  if (in_regs) {
#pragma unroll
    for (int j = 0; j < kRegUnits; ++j) {
      const int u = threadIdx.x + j * kNormThreads;
      v[j] = u < U ? rr[u] : make_float4(0.f, 0.f, 0.f, 0.f);
      ss = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, ss))));
    }
  } else {
    for (int u = threadIdx.x; u < U; u += kNormThreads) {
      const float4 x = rr[u];
      ss = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, ss))));
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)D + eps);
  auto put = [&](int u, const float4 x) {
    const uint2 gh = *reinterpret_cast<const uint2*>(gamma + 4 * u);
    const float2 g0 = __half22float2(u32_as_h2(gh.x)), g1 = __half22float2(u32_as_h2(gh.y));
    uint2 o;
    o.x = h2_as_u32(__floats2half2_rn(x.x * inv * g0.x, x.y * inv * g0.y));
    o.y = h2_as_u32(__floats2half2_rn(x.z * inv * g1.x, x.w * inv * g1.y));
    *reinterpret_cast<uint2*>(xn + row * D + 4 * u) = o;
  };
  if (in_regs) {
#pragma unroll
    for (int j = 0; j < kRegUnits; ++j) {
      const int u = threadIdx.x + j * kNormThreads;
      if (u < U) put(u, v[j]);
    }
  } else {
    for (int u = threadIdx.x; u < U; u += kNormThreads) put(u, rr[u]);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

template <int EPI>
cudaError_t launch_tc_t(const Launch& L, const TcMaps& m, const TcGemmArgs& a) {
  auto kern = tc_gemm_kernel<EPI>;
  const int smem = kGemmSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  static int n_sm = 0;
  if (!n_sm) {
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  }
  const int n_tiles = ((a.M + BM - 1) / BM) * (a.N / BN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(std::min(n_tiles, n_sm));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.counter) ++*L.counter;
  const CUtensorMap* ma = reinterpret_cast<const CUtensorMap*>(m.a);
  const CUtensorMap* mh = reinterpret_cast<const CUtensorMap*>(m.hi);
  const CUtensorMap* ml = reinterpret_cast<const CUtensorMap*>(m.lo);
  return cudaLaunchKernelEx(&cfg, kern, *ma, *mh, *ml, a);
}

}  // namespace

bool make_tmap_2d(void* map_out, const void* base, int64_t rows, int64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || (cols * 2) % 16 != 0 || (reinterpret_cast<uintptr_t>(base) & 15) != 0) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {BK, 128};
  cuuint32_t es[2] = {1, 1};
  return fn(reinterpret_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_gemm_rows_multiple() { return BN; }

cudaError_t launch_tc_gemm(const Launch& L, const TcMaps& m, const TcGemmArgs& a, int epi) {
  if (a.M < 1 || a.N < 1 || a.N % BN || a.K < 1) return cudaErrorInvalidValue;
  if (epi == EPI_RESID) return launch_tc_t<EPI_RESID>(L, m, a);
  if (epi == EPI_SWIGLU) return launch_tc_t<EPI_SWIGLU>(L, m, a);
  if (epi == EPI_QKV) return launch_tc_t<EPI_QKV>(L, m, a);
  return cudaErrorInvalidValue;
}

cudaError_t launch_rows_to_resid(const Launch& L, const __half* x, float* r, int T, int D) {
  if (T == 0) return cudaSuccess;
  rows_to_resid_kernel<<<T, 256, 0, L.stream>>>(x, r, D);
  if (L.counter) ++*L.counter;
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const Launch& L, const float* src, int D, const RowList& rows, float* dst) {
  if (rows.n < 1 || rows.n > MAG_MAX_BATCH) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows.n);
  cfg.blockDim = dim3(256);
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.counter) ++*L.counter;
  return cudaLaunchKernelEx(&cfg, gather_rows_kernel, src, D, rows, dst);
}

cudaError_t launch_rmsnorm_rows(const Launch& L, const float* r, const __half* gamma, float eps, int T, int D,
                                __half* xn) {
  if (T == 0) return cudaSuccess;
  if (D % 4) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T);
  cfg.blockDim = dim3(kNormThreads);
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.counter) ++*L.counter;
  return cudaLaunchKernelEx(&cfg, rmsnorm_rows_kernel, r, gamma, eps, D, xn);
}

}  // namespace mag
