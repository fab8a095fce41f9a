// Chunked prefill: the dense contractions of a T-token chunk on the 5th-generation
// tensor cores (tcgen05 MMA, accumulator in tensor memory, activations staged by TMA),
// plus the row-wise pieces around them.
//
// The chunk's projections are GEMMs Y[T][N] = X[T][K] W[N][K]^T over the W4 weights
// themselves ("5. Core modules" 5.1: 4-bit weights, FP16 activations): the GEMM
// reads the decode path's 640-byte tiles (16 rows x 64 k: codes, then fp16 (scale,
// min) pairs) and eight warps of every block expand each 128-row x 64-k slice of
// them into two fp16 operands in shared memory, hi = fp16(w) and lo = fp16(w - hi)
// of the exact w = s q + m (so hi + lo is w to 2^-22; one fp16 term alone rounds
// every weight, which 32 layers amplify past the parity bar), in the 128-byte-
// swizzled K-major layout the tensor core reads; every k-step accumulates X hi^T
// and X lo^T. One expanded slice serves two 128-token tiles, and the weights
// stream from HBM once per pair.
//
// GEMM block (persistent, one per SM): a unit is 128 weight rows x up to 256
// tokens (two 128-token tiles), K in steps of 64. Warp 0 issues the TMA loads of
// the activation tiles; warp 14 copies the W4 slices into a ring (cp.async.bulk)
// and warps 6-13 expand them into the weight operand; one thread of warp 1 issues
// tcgen05.mma (M 128 tokens, N 128 rows, K 16; fp32 in one of two 256-column
// halves of tensor memory) and commits each stage back; warps 2-5 read the
// accumulator with tcgen05.ld and run the epilogue while the next unit accumulates.
// Every wait is bounded; a role whose wait gives up sets its bit in the error word
// and drains what it has in flight (its copies, its MMAs) before the block frees
// its tensor memory and exits.
#include <cuda.h>

#include <algorithm>

#include "kernels.h"

namespace mag {

namespace {

constexpr int BM = 128, BN = 128, BK = 64, PT = 2;  // PT token tiles per unit
constexpr int TILE_A = BM * BK * 2, TILE_B = BN * BK * 2;
// three rings: activation tiles (TMA, from L2), expanded weights (written by the dequant warps from data
// already on chip, so a short ring), and the raw W4 slices (from HBM: the deepest, ~2 us of MMA work ahead)
constexpr int STAGES_A = 3, STAGES_B = 2;
constexpr int kDeqBatch = 1;  // k-steps a dequant warp expands per pass
constexpr int B_BYTES = 2 * TILE_B;  // a weight slice as two fp16 terms: hi, then lo
constexpr int A_BYTES = PT * TILE_A;
constexpr int kDeqWarps = 8, kDeqWarp0 = 6;           // warps 6..13 expand the weights, one decode tile each
constexpr int kLoadWarp = kDeqWarp0 + kDeqWarps;      // warp 14 copies the raw W4 slices
constexpr int kRawSlots = 6;                           // ring of raw W4 slices
constexpr int kRawBytes = 8 * kTileBytes;              // the 8 decode tiles of one 128-row x 64-k slice
constexpr int kGemmThreads = (kLoadWarp + 1) * 32;
constexpr int kTmemCols = 2 * PT * BN;                 // two units' accumulators

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void mb_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mb_expect(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mb_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
// One poll: the thread may sleep until the phase completes or up to ~1 us (the suspend-time hint), so that
// waiting warps leave the issue slots to the working ones.
__device__ __forceinline__ bool mb_try(uint64_t* b, uint32_t par) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(par)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of parity `par`: at most `limit` polls.
__device__ __forceinline__ bool mb_wait(uint64_t* b, uint32_t par, uint32_t limit = kWaitPolls) {
  for (uint32_t i = 0; i < limit; ++i)
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
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(bar))
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
__device__ __forceinline__ void tmem_ld32_raw(uint32_t taddr, float (&v)[32]) {
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

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// Eight codes of one word (nibble i = element i) with the group's (scale, min) -> the eight weights
// w = s q + m as two fp16 terms in element order: w in fp32 (s q is exact, one rounding for + m: the
// format's dequantised value), hi = fp16(w), lo = fp16(w - hi), so hi + lo is w to 2^-22. Nibble pairs
// (i, i + 4) become fp16 1024 + q by mask-and-or (1024 subtracted exactly), and the pairs are put back
// in element order at the end.
__device__ __forceinline__ void dequant8_hilo(uint32_t w, uint32_t sm, uint4& hi, uint4& lo) {
  const float2 sf = __half22float2(u32_as_h2(sm));  // (scale, min)
  const __half2 k1024 = u32_as_h2(0x64006400u);
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t qb = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;
    const float2 q = __half22float2(__hsub2(u32_as_h2(qb), k1024));  // codes (i, i + 4), exact
    const float w0 = fmaf(sf.x, q.x, sf.y), w1 = fmaf(sf.x, q.y, sf.y);
    const __half2 hh = __floats2half2_rn(w0, w1);
    const float2 hf = __half22float2(hh);
    h[i] = h2_as_u32(hh);
    l[i] = h2_as_u32(__floats2half2_rn(w0 - hf.x, w1 - hf.y));
  }
  hi = make_uint4(prmt(h[0], h[1], 0x5410), prmt(h[2], h[3], 0x5410), prmt(h[0], h[1], 0x7632), prmt(h[2], h[3], 0x7632));
  lo = make_uint4(prmt(l[0], l[1], 0x5410), prmt(l[2], l[3], 0x5410), prmt(l[0], l[1], 0x7632), prmt(l[2], l[3], 0x7632));
}

__device__ __forceinline__ float silu_mul(float gte, float up) { return gte / (1.0f + expf(-gte)) * up; }

constexpr int kSq = 36;                              // floats per staged row (see the epilogue)
constexpr int kStageSqBytes = 32 * kSq * 4;          // one warp's 32 x 32 staging square
constexpr int kBarBytes = 512;  // 31 mbarriers and the TMEM address
constexpr int kRingBytes = STAGES_A * A_BYTES + STAGES_B * B_BYTES;
constexpr int kGemmSmem = kRingBytes + kRawSlots * kRawBytes + 4 * kStageSqBytes + kBarBytes + 1024;

// Persistent: one block per SM takes units u = blockIdx.x + i gridDim.x; unit u is weight tile u / n_pairs
// (128 GEMM rows) x token tiles 2 (u % n_pairs), +1 (the token pairs of a weight tile are launch-order
// neighbours, so its W4 bytes come from HBM once). The stage ring runs on across units and the
// accumulators are double-buffered in tensor memory, so the epilogue of unit i overlaps unit i + 1.
template <int EPI>
__global__ void __launch_bounds__(kGemmThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const TcGemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_ring = smem;                                  // [STAGES_A][PT][128 x 64 fp16]
  uint8_t* b_ring = smem + STAGES_A * A_BYTES;             // [STAGES_B][hi, lo][128 x 64 fp16]
  uint8_t* raw = smem + kRingBytes;
  float* stage_sq = reinterpret_cast<float*>(raw + kRawSlots * kRawBytes);
  uint64_t* a_full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(stage_sq) + 4 * kStageSqBytes);
  uint64_t* a_empty = a_full + STAGES_A;
  uint64_t* b_full = a_empty + STAGES_A;
  uint64_t* b_empty = b_full + STAGES_B;
  uint64_t* acc_full = b_empty + STAGES_B;           // [2]
  uint64_t* acc_empty = acc_full + 2;                // [2]
  uint64_t* raw_full = acc_empty + 2;                // [kRawSlots]
  uint64_t* raw_empty = raw_full + kRawSlots;        // [kRawSlots]
  uint64_t* mma_done = raw_empty + kRawSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_m = (a.M + BM - 1) / BM, n_pairs = (n_m + PT - 1) / PT;
  // unit u: output block ub = u / S (weight tile ub / n_pairs x token pair ub % n_pairs) and K half u % S
  const int S = a.ksplit, n_units = n_pairs * (a.N / BN) * S;
  const int nks = (a.K + BK - 1) / BK / S;  // k-steps of one unit (the host makes S divide them)
  auto unit_tiles = [&](int u) { return min(PT, n_m - ((u / S) % n_pairs) * PT); };  // token tiles of unit u
  auto unit_kb0 = [&](int u) { return (u % S) * nks; };
  auto unit_wt = [&](int u) { return (u / S) / n_pairs; };
  auto unit_m0 = [&](int u) { return ((u / S) % n_pairs) * PT * BM; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES_A; ++s) {
      mb_init(a_full + s, 1);
      mb_init(a_empty + s, 1);
    }
    for (int s = 0; s < STAGES_B; ++s) {
      mb_init(b_full + s, kDeqWarps);
      mb_init(b_empty + s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mb_init(acc_full + i, 1);
      mb_init(acc_empty + i, 4);  // one arrival per epilogue warp
    }
    for (int i = 0; i < kRawSlots; ++i) {
      mb_init(raw_full + i, 1);
      mb_init(raw_empty + i, kDeqWarps);
    }
    mb_init(mma_done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer of the activation tiles (they come from the previous kernel)
    if (lane == 0) {
      pdl_wait();
      int g = 0;  // stages issued so far, over all units
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const int nt = unit_tiles(u), m0 = unit_m0(u);
        for (int kb = unit_kb0(u); kb < unit_kb0(u) + nks; ++kb, ++g) {
          const int s = g % STAGES_A;
          if (g >= STAGES_A && !mb_wait(a_empty + s, ((g / STAGES_A) - 1) & 1, a.wait_limit)) {
            atomicOr(a.err, 8u);
            ok = false;
            break;
          }
          uint8_t* st = a_ring + s * A_BYTES;
          mb_expect(a_full + s, nt * TILE_A);
          for (int p = 0; p < nt; ++p) tma_2d(st + p * TILE_A, &map_a, kb * BK, m0 + p * BM, a_full + s);
        }
      }
      // leave no copy in flight, also when a consumer gave up and will not wait for them: the last load of
      // every slot has landed (at once on the normal path, where the MMA thread has waited for them)
      for (int f = max(0, g - STAGES_A); f < g; ++f) mb_wait(a_full + f % STAGES_A, (f / STAGES_A) & 1);
    }
  } else if (warp == kLoadWarp) {
    // ---- raw W4 slices: the 8 decode tiles of a unit's weight tile at k-step kb (640 bytes each, one bulk
    // copy per tile) into the ring, kRawSlots stages ahead of the expansion; the weights do not depend on
    // earlier kernels. A thread of its own issues them: a proxy fence in a warp with its own bulk copies in
    // flight would wait for those copies.
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const int jg = unit_wt(u) * 8, nv = max(0, min(8, a.n_dtiles - jg));
        for (int kb = unit_kb0(u); kb < unit_kb0(u) + nks; ++kb, ++g) {
          const int r = g % kRawSlots;
          if (g >= kRawSlots && !mb_wait(raw_empty + r, ((g / kRawSlots) - 1) & 1, a.wait_limit)) {
            atomicOr(a.err, 256u);
            ok = false;
            break;
          }
          uint8_t* dst = raw + r * kRawBytes;
          mb_expect(raw_full + r, nv * kTileBytes);
          for (int j = 0; j < nv; ++j)
            bulk_g2s(dst + j * kTileBytes, a.w + ((int64_t)(jg + j) * a.C + kb) * kTileBytes, kTileBytes,
                     raw_full + r);
        }
      }
      // leave no copy in flight, also when the expansion gave up and will not wait for them
      for (int f = max(0, g - kRawSlots); f < g; ++f) mb_wait(raw_full + f % kRawSlots, (f / kRawSlots) & 1);
    }
  } else if (warp >= kDeqWarp0) {
    // ---- W4 expansion: this warp's decode tile (16 rows) of every 128-row x 64-k slice, two slices per pass
    // (one proxy fence and one round of barriers for both, twice the independent work between them). Lane
    // (g, t) holds word t of rows g and g+8 for the slice's two 32-groups; GEMM row of tile-row (j, g, h):
    // (j / tpg) gsz + 8 (j % tpg) + g + h half
    const int wq = warp - kDeqWarp0, g8 = lane >> 2, t = lane & 3;
    const int my_units = blockIdx.x < n_units ? (n_units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int n_stages = my_units * nks;
    const int n_lo = (wq / a.tpg) * a.gsz + 8 * (wq % a.tpg) + g8;  // row of tile-row (wq, g, 0)
    bool ok = true;
    for (int g0 = 0; g0 < n_stages && ok; g0 += kDeqBatch) {
      const int nb = min(kDeqBatch, n_stages - g0);
      uint4 cw[kDeqBatch], sm[kDeqBatch];
      bool live[kDeqBatch];
#pragma unroll
      for (int e = 0; e < kDeqBatch; ++e) {
        if (e >= nb) break;
        const int g = g0 + e, r = g % kRawSlots;
        const int u = blockIdx.x + (g / nks) * gridDim.x;
        live[e] = unit_wt(u) * 8 + wq < a.n_dtiles;
        if (!__all_sync(0xffffffffu, mb_wait(raw_full + r, (g / kRawSlots) & 1, a.wait_limit))) {
          if (lane == 0) atomicOr(a.err, 128u);
          ok = false;
          break;
        }
        const uint8_t* rs = raw + r * kRawBytes + wq * kTileBytes;
        cw[e] = *reinterpret_cast<const uint4*>(rs + lane * 16);
        sm[e] = *reinterpret_cast<const uint4*>(rs + 512 + g8 * 16);
      }
      if (!ok) break;
      // the slots are in registers: release them to the loader (its wait orders the refills after these reads)
      __syncwarp();
      if (lane == 0)
        for (int e = 0; e < nb; ++e) mb_arrive(raw_empty + (g0 + e) % kRawSlots);
#pragma unroll
      for (int e = 0; e < kDeqBatch; ++e) {
        if (e >= nb) break;
        const int g = g0 + e;
        if (g >= STAGES_B &&
            !__all_sync(0xffffffffu, mb_wait(b_empty + g % STAGES_B, ((g / STAGES_B) - 1) & 1, a.wait_limit))) {
          if (lane == 0) atomicOr(a.err, 128u);
          ok = false;
          break;
        }
      }
      if (!ok) break;
#pragma unroll
      for (int e = 0; e < kDeqBatch; ++e) {
        if (e >= nb) break;
        uint8_t* bt = b_ring + ((g0 + e) % STAGES_B) * B_BYTES;
        const uint32_t words[4] = {cw[e].x, cw[e].y, cw[e].z, cw[e].w};  // (row g | g+8) x (group 0 | 1)
        const uint32_t sms[4] = {sm[e].x, sm[e].y, sm[e].z, sm[e].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int h = q >> 1, grp = q & 1;
          const int n = n_lo + h * a.half, c16 = 4 * grp + t;
          uint4 hi = make_uint4(0, 0, 0, 0), lo = hi;
          if (live[e]) dequant8_hilo(words[q], sms[q], hi, lo);
          const int off = n * 128 + ((c16 ^ (n & 7)) << 4);
          *reinterpret_cast<uint4*>(bt + off) = hi;
          *reinterpret_cast<uint4*>(bt + TILE_B + off) = lo;
        }
      }
      // the generic-proxy stores must be visible to the tensor core's (async-proxy) reads
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0)
        for (int e = 0; e < nb; ++e) mb_arrive(b_full + (g0 + e) % STAGES_B);
    }
  } else if (warp == 1) {
    // ---- MMA issuer: unit i into accumulator half i % 2, once the epilogue has drained it
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int u = blockIdx.x, it = 0; u < n_units && ok; u += gridDim.x, ++it) {
        const int ab = it & 1, nt = unit_tiles(u);
        if (it >= 2 && !mb_wait(acc_empty + ab, ((it >> 1) - 1) & 1, a.wait_limit)) {
          atomicOr(a.err, 64u);
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d = tmem + (uint32_t)(ab * PT * BN);
        for (int kb = 0; kb < nks; ++kb, ++g) {
          const int sa = g % STAGES_A, sb = g % STAGES_B;
          if (!mb_wait(a_full + sa, (g / STAGES_A) & 1, a.wait_limit) ||
              !mb_wait(b_full + sb, (g / STAGES_B) & 1, a.wait_limit)) {
            atomicOr(a.err, 16u);
            ok = false;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          uint8_t* st = a_ring + sa * A_BYTES;
          const uint64_t dh = smem_desc(b_ring + sb * B_BYTES), dl = smem_desc(b_ring + sb * B_BYTES + TILE_B);
          for (int p = 0; p < nt; ++p) {
            const uint64_t da = smem_desc(st + p * TILE_A);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint64_t off = (uint64_t)(k * 32) >> 4;  // 16 fp16 further along K
              mma_f16(d + (uint32_t)(p * BN), da + off, dh + off, (kb | k) != 0);
              mma_f16(d + (uint32_t)(p * BN), da + off, dl + off, 1);
            }
          }
          mma_commit(a_empty + sa);
          mma_commit(b_empty + sb);
        }
        if (ok) mma_commit(acc_full + ab);
      }
      // every MMA this thread issued has completed before the block frees its tensor memory
      mma_commit(mma_done);
      mb_wait(mma_done, 0);
    }
  } else {
    // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 = rows of a token tile. A thread holds one
    // row; the warp passes each 32-column slice through its own padded shared-memory square so that
    // global memory sees whole 16-byte runs of a row.
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
    for (int u = blockIdx.x, it = 0; u < n_units; u += gridDim.x, ++it) {
      const int ab = it & 1, nt = unit_tiles(u);
      const int n0 = unit_wt(u) * BN;
      if (!mb_wait(acc_full + ab, (it >> 1) & 1, a.wait_limit)) {
        atomicOr(a.err, 32u);
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      // K split in halves: each half leaves this warp's 32 rows of its partial sums in the workspace
      // ([half][token tile][column][lane]); the second to arrive adds the other half's to its own (a + b:
      // the same bits in either order) and runs the epilogue, the first is done.
      const float* other = nullptr;
      if (S > 1) {
        const int ub = u / S, kh = u % S;
        float* blk = a.part + (size_t)(ub * 4 + q) * S * PT * BN * 32;
        for (int p = 0; p < nt; ++p) {
          const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)((ab * PT + p) * BN);
          float* mine = blk + ((size_t)kh * PT + p) * BN * 32;
          for (int c0 = 0; c0 < BN; c0 += 32) {
            float v[32];
            tmem_ld32_raw(trow + c0, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) __stcg(mine + (c0 + j) * 32 + lane, v[j]);
          }
        }
        __threadfence();
        __syncwarp();
        uint32_t prev = 0;
        if (lane == 0) prev = atomicAdd(a.part_cnt + ub * 4 + q, 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if ((int)prev + 1 < S) {  // the other half is still running: it finishes the block
          asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
          __syncwarp();
          if (lane == 0) mb_arrive(acc_empty + ab);
          continue;
        }
        __threadfence();
        if (lane == 0) a.part_cnt[ub * 4 + q] = 0;  // for the next launch
        other = blk + (size_t)(1 - kh) * PT * BN * 32;
      }
      for (int p = 0; p < nt; ++p) {
        const int m0 = unit_m0(u) + p * BM;
        const int m = m0 + q * 32 + lane, row0 = m0 + q * 32;
        const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)((ab * PT + p) * BN);
        const float* oth = other ? other + (size_t)p * BN * 32 : nullptr;
        // 32 accumulator columns from c of this lane's row, plus the other K half's partial sums
        auto tmem_ld32 = [&](uint32_t taddr, float (&v)[32]) {
          mag::tmem_ld32_raw(taddr, v);
          if (oth) {
            const int c = (int)(taddr - trow);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += __ldcg(oth + (c + j) * 32 + lane);
          }
        };
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
            float gv[32], uv[32];
            tmem_ld32(trow + c0, gv);
            tmem_ld32(trow + c0 + BN / 2, uv);
#pragma unroll
            for (int j = 0; j < 32; ++j) gv[j] = silu_mul(gv[j], uv[j]);
            put_row(gv);
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
            if (i0 >= hd || n0 + c0 >= a.n_valid) continue;  // second halves come with the first; padding rows
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
      }
      // the accumulator half is drained: the MMA warp may reuse it
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mb_arrive(acc_empty + ab);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
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
cudaError_t launch_tc_t(const Launch& L, const void* map_a, const TcGemmArgs& a) {
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
  const int n_m = (a.M + BM - 1) / BM, n_units = ((n_m + PT - 1) / PT) * (a.N / BN) * a.ksplit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(std::min(n_units, n_sm));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L.counter) ++*L.counter;
  return cudaLaunchKernelEx(&cfg, kern, *reinterpret_cast<const CUtensorMap*>(map_a), a);
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

int tc_gemm_ksplit(int M, int N, int K, int n_sm) {
  const int n_m = (M + BM - 1) / BM, base = ((n_m + PT - 1) / PT) * (N / BN), nk = (K + BK - 1) / BK;
  return 2 * base <= n_sm && nk % 2 == 0 ? 2 : 1;
}

size_t tc_gemm_part_floats(int n_sm) { return (size_t)(n_sm / 2) * 4 * 2 * PT * BN * 32; }

cudaError_t launch_tc_gemm(const Launch& L, const void* map_a, const TcGemmArgs& a, int epi) {
  if (a.M < 1 || a.N < 1 || a.N % BN || a.K < 1 || !a.w || a.n_dtiles < 1 || a.n_dtiles > a.N / 16 ||
      a.C != (a.K + BK - 1) / BK || a.tpg < 1 || a.tpg > 8 || a.half < 8 || a.ksplit < 1 || a.ksplit > 2 ||
      a.C % a.ksplit || (a.ksplit > 1 && (!a.part || !a.part_cnt)))
    return cudaErrorInvalidValue;
  if (epi == EPI_RESID) return launch_tc_t<EPI_RESID>(L, map_a, a);
  if (epi == EPI_SWIGLU) return launch_tc_t<EPI_SWIGLU>(L, map_a, a);
  if (epi == EPI_QKV) return launch_tc_t<EPI_QKV>(L, map_a, a);
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
