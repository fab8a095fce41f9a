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
// score scale. The blocks of one (session, KV head) form a thread-block
// cluster; each streams its share of the pool blocks through a per-warp
// cp.async ring in shared memory, and the cluster merges its split partials
// (m, l, o) through distributed shared memory.
#include <cooperative_groups.h>

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
  if ((unsigned)blk >= (unsigned)a.pool.pool_blocks) {  // a table entry outside the pool: store nothing
    if (i == 0 && a.err) atomicOr(a.err, kErrBounds);
    return;
  }
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

// ---------------------------------------------------------------- attention
// Shared-memory image of one (block, KV head): K data [16][db], V data [16][db],
// K meta [16][mb], V meta [16][mb], each region 16-byte aligned.
template <int D, int DT>
struct SlotGeom {
  static constexpr int kDb = DT == 0 ? 2 * D : (DT == 1 ? D : D / 2);     // bytes per K or V vector
  static constexpr int kMb = DT == 0 ? 0 : (DT == 1 ? 2 : (D / 32) * 4);  // meta bytes per vector
  static constexpr int kData = 16 * kDb;
  static constexpr int kMeta = ((16 * kMb) + 15) / 16 * 16;
  static constexpr int kBytes = 2 * kData + 2 * kMeta;
};

__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Copy one (block, KV head) of the pool into a slot (the 32 lanes of a warp, 16 bytes each).
template <int D, int DT>
__device__ __forceinline__ void issue_block(uint8_t* slot, const PoolGeom& P, int layer, int phys, int gk, int lane) {
  using SG = SlotGeom<D, DT>;
  const uint8_t* kd = pool_vec(P, layer, phys, 0, gk, 0);
  const uint8_t* vd = pool_vec(P, layer, phys, 1, gk, 0);
#pragma unroll
  for (int o = lane * 16; o < SG::kData; o += 512) {
    cp_async16(slot + o, kd + o);
    cp_async16(slot + SG::kData + o, vd + o);
  }
  if (DT != 0) {
    const uint8_t* km = pool_vec(P, layer, phys, 2, gk, 0);
    const uint8_t* vm = pool_vec(P, layer, phys, 3, gk, 0);
    constexpr int mbytes = 16 * SG::kMb;
    for (int o = lane * 16; o < mbytes; o += 512) {
      cp_async16(slot + 2 * SG::kData + o, km + o);
      cp_async16(slot + 2 * SG::kData + SG::kMeta + o, vm + o);
    }
  }
}

// V dims of lane group gi for one token: NV halves as NV/2 words, slot order.
template <int D, int DT>
__device__ __forceinline__ void load_v_row(const uint8_t* row, const uint8_t* meta, int gi, uint32_t (&out)[D / 16]) {
  constexpr int NV = D / 8;
  if (DT == 0) {
    const uint4* p = reinterpret_cast<const uint4*>(row + gi * NV * 2);
#pragma unroll
    for (int j = 0; j < NV / 8; ++j) {
      const uint4 v = p[j];
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
    const __half2 sm = *reinterpret_cast<const __half2*>(meta + 4 * ((gi * NV) / 32));
#pragma unroll
    for (int j = 0; j < NV / 8; ++j) {
      const uint4 o = u4x8_to_h2(p[j], sm);
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

// The 8 x 8 fp16 matrix held one row pair per lane (lane 4 r + c: row r, columns 2c, 2c+1), transposed.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
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

constexpr int kAttnSlots = 3;  // per-warp ring depth, in (block, KV head) units

// Shared-memory image of the NW warps' partial outputs [warp][head (8)][dim] and the block's merged partial
// o [head][dim]; both reuse the rings' shared memory once every warp has left its loop.
template <int D, int NW>
struct AccGeom {
  static constexpr size_t kAccBytes = (size_t)NW * 8 * D * 4;
  static constexpr size_t kBytes = kAccBytes + (size_t)8 * D * 4;  // + the partial o
};

template <int D, int DT, int NW>
__host__ __device__ constexpr size_t attn_smem_bytes() {
  return (size_t)NW * kAttnSlots * SlotGeom<D, DT>::kBytes > AccGeom<D, NW>::kBytes
             ? (size_t)NW * kAttnSlots * SlotGeom<D, DT>::kBytes
             : AccGeom<D, NW>::kBytes;
}

// Warps per block of the wide variant (long contexts: more warps per SM to hide the per-block chain).
// At head_dim 128 a lane holds ~185 registers, so 4-warp blocks stop at two per SM (8 warps) and 16-warp
// blocks would spill under the 128-register cap: 8 warps, one block per SM on every SM of the grid.
// At head_dim 64, 16 warps where their rings fit one SM's shared memory.
template <int D, int DT>
constexpr int attn_wide_warps() {
  return D > 64 ? 8 : ((size_t)16 * kAttnSlots * SlotGeom<D, DT>::kBytes <= 220 * 1024 ? 16 : 8);
}

// The last block of a (row, KV head) to arrive: its K parts' (m, l, o) of the G d outputs combined in part
// order into out. Kept out of line, so that its registers do not weigh on the attention kernel's loop.
__device__ __noinline__ void merge_parts(const float* pb, int K, int GD, __half* out) {
  for (int idx = threadIdx.x; idx < GD; idx += blockDim.x) {
    // all K parts in flight at once (one round trip)
    float mq[kAttnMaxGroups], lq[kAttnMaxGroups], oq[kAttnMaxGroups];
#pragma unroll
    for (int q = 0; q < kAttnMaxGroups; ++q) {
      const float* pq = pb + (int64_t)q * 3 * GD;
      const bool v = q < K;
      mq[q] = v ? __ldcg(pq + idx) : -INFINITY;
      lq[q] = v ? __ldcg(pq + GD + idx) : 0.f;
      oq[q] = v ? __ldcg(pq + 2 * GD + idx) : 0.f;
    }
    float mm = -INFINITY;
#pragma unroll
    for (int q = 0; q < kAttnMaxGroups; ++q) mm = fmaxf(mm, mq[q]);
    float l = 0.f, o = 0.f;
#pragma unroll
    for (int q = 0; q < kAttnMaxGroups; ++q) {
      const float e = mq[q] == -INFINITY ? 0.f : exp2f(mq[q] - mm);
      l = fmaf(lq[q], e, l);
      o = fmaf(oq[q], e, o);
    }
    out[idx] = __float2half_rn(o / l);
  }
}

// One block of the grid per (split, KV head, session); the blocks of a
// (session, KV head) form a thread-block cluster and merge their splits
// through distributed shared memory. NWARP warps per block.
template <int D, int DT, int NWARP>
__global__ void __launch_bounds__(32 * NWARP, NWARP <= 4 ? 4 : (NWARP <= 8 ? 2 : 1)) attn_kernel(const AttnArgs a) {
  namespace cg = cooperative_groups;
  using SG = SlotGeom<D, DT>;
  using AG = AccGeom<D, NWARP>;
  constexpr int NS = D / 32;  // 32-dim slabs of K (one INT4 group each)
  constexpr int NV = D / 8;   // V n-tiles
  constexpr int NW = D / 16;  // words per V row of a lane
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_m[NWARP][8], s_l[NWARP][8];
  float* s_acc = reinterpret_cast<float*>(smem);                    // after the loops
  float* s_po = reinterpret_cast<float*>(smem + AG::kAccBytes);      // this block's partial o [head][dim]
  __shared__ float s_pm[8], s_pl[8];  // this block's partial (m, l) per head
  __shared__ __half s_kv[2][D];
  __shared__ float s_red[8];
  // inbox of the cluster merge: every rank's partial o of this rank's share of the outputs, [rank][share],
  // and every rank's (m, l) per head
  __shared__ __align__(16) float s_in_o[8 * D + 16];
  __shared__ float s_in_m[16][8], s_in_l[16][8];

  cg::cluster_group cluster = cg::this_cluster();
  // the first half of a split barrier: its wait (before the first store into another rank's shared memory)
  // then only confirms that every block of the cluster has started
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  const int split = blockIdx.x, gk = blockIdx.y, b = blockIdx.z;
  // step timeline stamps (the tag rebuilt from the arguments at each, so that nothing stays live)
  auto stamp = [&](unsigned int ev) { trace_stamp(a.trace, kTraceAttn | (unsigned)a.layer, ev); };
  if (threadIdx.x == 0) stamp(0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gi = lane >> 2, t = lane & 3;
  const int Hq = a.n_heads, Hkv = a.n_kv_heads, G = Hq / Hkv;
  const int S = a.n_split;  // == cluster size
  const int K = a.n_groups;  // clusters per (session, KV head); S K splits in all, blockIdx.x = split
  // The step's arguments were copied before the step's first kernel and the
  // pool blocks before the new token's were written and mapped by earlier
  // steps, so their fetch starts before waiting for the QKV projection.
  const int pos = a.step->pos[b], sess = a.step->sess[b];
  const int n_keys = pos + 1, new_blk = pos >> 4;
  // blocks from fresh_blk on hold keys written in this step (the row's own, or with stored keys those of
  // the session's earlier rows as well); they are mapped and fetched only after the wait
  const int fresh_blk = a.stored == 1 ? a.step->pos[0] >> 4 : new_blk;
  const int n_blocks = new_blk + 1;
  const int bps = (n_blocks + S * K - 1) / (S * K);
  const int blk0 = split * bps, blk1 = min(blk0 + bps, n_blocks);
  const int32_t* table = a.pool.tables + (int64_t)sess * a.pool.table_stride;
  // this warp's blocks: blk0 + warp + NWARP j; the new token's block, if it is one
  // of them, is the last
  const int nb = blk0 + warp < blk1 ? (blk1 - blk0 - warp + NWARP - 1) / NWARP : 0;
  // physical ids of the warp's first 32 blocks, one lane each (one round trip for all of them); a block
  // from fresh_blk on may have been mapped by this step's prologue, so its id is read after the wait
  const int phys_l = lane < nb ? table[blk0 + warp + NWARP * lane] : 0;
  int phys_new = -1;
  auto phys_of = [&](int j) {
    const int blk = blk0 + warp + NWARP * j;
    const int p = j < 32 ? __shfl_sync(0xffffffffu, phys_l, j) : table[blk];
    // an id outside the pool (a corrupted table) is not used: block 0 instead, and the error word says so
    return checked_block(blk == new_blk ? phys_new : blk >= fresh_blk ? table[blk] : p, a.pool.pool_blocks, a.err);
  };
  uint8_t* ring = smem + (size_t)warp * kAttnSlots * SG::kBytes;
  int issued = 0;
  for (; issued < min(nb, kAttnSlots); ++issued) {
    const int blk = blk0 + warp + NWARP * issued;
    if (blk >= fresh_blk) break;
    issue_block<D, DT>(ring + issued * SG::kBytes, a.pool, a.layer, phys_of(issued), gk, lane);
    cp_async_commit();
  }
  phys_new = a.step->blk[b];  // the host's copy of table[new_blk]: no table read after the wait
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) stamp(1);
  const __half* qkv = a.qkv + (int64_t)b * a.qkv_ld;

  // the block that holds the new token appends its K (rotated) and V to the pool
  if (a.stored == 0 && blk0 <= new_blk && new_blk < blk1) {
    if (tid < D) {
      s_kv[0][tid] = qkv[(int64_t)(Hq + gk) * D + tid];
      s_kv[1][tid] = qkv[(int64_t)(Hq + Hkv + gk) * D + tid];
    }
    __syncthreads();
    const int phys = phys_new;
    store_vec(a.pool, a.layer, phys, pos & 15, gk, 0, s_kv[0], s_red);
    store_vec(a.pool, a.layer, phys, pos & 15, gk, 1, s_kv[1], s_red);
    __threadfence_block();
    __syncthreads();
  }
  // this warp's deferred fetches: the ring slots its blocks from fresh_blk on did not get before the wait
  for (; issued < min(nb, kAttnSlots); ++issued) {
    issue_block<D, DT>(ring + issued * SG::kBytes, a.pool, a.layer, phys_of(issued), gk, lane);
    cp_async_commit();
  }
  for (; issued < kAttnSlots; ++issued) cp_async_commit();  // one group per ring slot

  // The heads are the MMAs' 8 columns (G <= 8 of them; zero queries past G) and the block's 16 tokens, or
  // the head's dims, the 16 rows: S^T = K Q^T and O^T += V^T P^T, so no MMA row is padding.
  // Query B fragments: lane (gi, t) holds head gi's dims 32 s + 8 t .. + 7 of slab s (INT4: in the codes'
  // (k0,k4) (k1,k5) (k2,k6) (k3,k7) order), the k-slots of the slab's two k-steps.
  uint32_t qb[2 * NS][2];
  float qsum[NS];  // INT4: per 32-dim slab, the sum of head gi's query values
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
    qb[2 * s][0] = v.x;
    qb[2 * s][1] = v.y;
    qb[2 * s + 1][0] = v.z;
    qb[2 * s + 1][1] = v.w;
  }
  // INT4: the query sums of heads 2t and 2t+1, the columns of this lane's score fragments
  float qs2[NS][2];
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    qs2[s][0] = __shfl_sync(0xffffffffu, DT == 2 ? qsum[s] : 0.f, 8 * t);
    qs2[s][1] = __shfl_sync(0xffffffffu, DT == 2 ? qsum[s] : 0.f, 8 * t + 4);
  }
  const float sc = 1.4426950408889634f / sqrtf((float)D);  // log2(e) / sqrt(d)
  // running maximum and sum of heads 2t, 2t+1; acc[m] = O^T rows g, g+8 of m-tile m (dims of slots 2m, 2m+1
  // of lane group gi) x columns 2t, 2t+1 (heads)
  float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};
  float acc[NV / 2][4];
#pragma unroll
  for (int m = 0; m < NV / 2; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;

  int slot_i = 0;
  for (int j = 0; j < nb; ++j) {
    const int blk = blk0 + warp + NWARP * j;
    uint8_t* slot = ring + slot_i * SG::kBytes;
    cp_async_wait<kAttnSlots - 1>();
    __syncwarp();
    const uint8_t* kd = slot;
    const uint8_t* vd = slot + SG::kData;
    const uint8_t* km = slot + 2 * SG::kData;
    const uint8_t* vm = km + SG::kMeta;
    // ---- scores S^T[token][head]: rows gi, gi+8 of the block's tokens, columns 2t, 2t+1; the slabs in two
    // independent accumulation chains
    const uint8_t* kr0 = kd + gi * SG::kDb;
    const uint8_t* kr8 = kd + (gi + 8) * SG::kDb;
    float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (DT == 2) {
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const uint4 k0 = u4x8_codes(*reinterpret_cast<const uint32_t*>(kr0 + 16 * s + 4 * t));
        const uint4 k8 = u4x8_codes(*reinterpret_cast<const uint32_t*>(kr8 + 16 * s + 4 * t));
        float as[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(as, k0.x, k8.x, k0.y, k8.y, qb[2 * s][0], qb[2 * s][1]);
        mma_16816(as, k0.z, k8.z, k0.w, k8.w, qb[2 * s + 1][0], qb[2 * s + 1][1]);
        // per (token, group): score += s * (codes . q) + m * sum(q)
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(km + gi * SG::kMb + 4 * s));
        const float2 f8 = __half22float2(*reinterpret_cast<const __half2*>(km + (gi + 8) * SG::kMb + 4 * s));
        float* acc_s = s2[s & 1];
        acc_s[0] = fmaf(f0.x, as[0], fmaf(f0.y, qs2[s][0], acc_s[0]));
        acc_s[1] = fmaf(f0.x, as[1], fmaf(f0.y, qs2[s][1], acc_s[1]));
        acc_s[2] = fmaf(f8.x, as[2], fmaf(f8.y, qs2[s][0], acc_s[2]));
        acc_s[3] = fmaf(f8.x, as[3], fmaf(f8.y, qs2[s][1], acc_s[3]));
      }
    } else {
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        uint4 k0, k8;
        if (DT == 0) {
          k0 = *reinterpret_cast<const uint4*>(kr0 + (32 * s + 8 * t) * 2);
          k8 = *reinterpret_cast<const uint4*>(kr8 + (32 * s + 8 * t) * 2);
        } else {
          const uint2 w0 = *reinterpret_cast<const uint2*>(kr0 + 32 * s + 8 * t);
          const uint2 w8 = *reinterpret_cast<const uint2*>(kr8 + 32 * s + 8 * t);
          i8x4_to_h2(w0.x, k0.x, k0.y);
          i8x4_to_h2(w0.y, k0.z, k0.w);
          i8x4_to_h2(w8.x, k8.x, k8.y);
          i8x4_to_h2(w8.y, k8.z, k8.w);
        }
        mma_16816(s2[s & 1], k0.x, k8.x, k0.y, k8.y, qb[2 * s][0], qb[2 * s][1]);
        mma_16816(s2[s & 1], k0.z, k8.z, k0.w, k8.w, qb[2 * s + 1][0], qb[2 * s + 1][1]);
      }
    }
    // e: 0 (token gi, head 2t), 1 (gi, 2t+1), 2 (gi+8, 2t), 3 (gi+8, 2t+1)
    float sfr[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) sfr[e] = s2[0][e] + s2[1][e];
    float ks[2] = {1.f, 1.f}, vsc[2] = {1.f, 1.f};  // INT8 scales of tokens gi, gi+8
    if (DT == 1) {
      ks[0] = __half2float(*reinterpret_cast<const __half*>(km + gi * 2));
      ks[1] = __half2float(*reinterpret_cast<const __half*>(km + (gi + 8) * 2));
      vsc[0] = __half2float(*reinterpret_cast<const __half*>(vm + gi * 2));
      vsc[1] = __half2float(*reinterpret_cast<const __half*>(vm + (gi + 8) * 2));
    }
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int tok = blk * 16 + gi + 8 * (e >> 1);
      const float v = tok < n_keys ? sfr[e] * ks[e >> 1] * sc : -INFINITY;
      sfr[e] = v;
      mx[e & 1] = fmaxf(mx[e & 1], v);
    }
    float corr[2], m_new[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 4));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 8));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 16));
      m_new[h] = fmaxf(m_run[h], mx[h]);
      corr[h] = exp2f(m_run[h] - m_new[h]);
      m_run[h] = m_new[h];
    }
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = exp2f(sfr[e] - m_new[e & 1]);
    l_part[0] = l_part[0] * corr[0] + p[0] + p[2];
    l_part[1] = l_part[1] * corr[1] + p[1] + p[3];
#pragma unroll
    for (int m = 0; m < NV / 2; ++m) {
      acc[m][0] *= corr[0];
      acc[m][1] *= corr[1];
      acc[m][2] *= corr[0];
      acc[m][3] *= corr[1];
    }
    // P^T (times the INT8 value scale) as the B operand, split into fp16 hi + lo so the product carries no
    // fp16 rounding of the probabilities: the 8 x 8 tiles [token][head] of tokens 0-7 and 8-15, transposed
    // in registers into [head][token] (b0: tokens 2t, 2t+1; b1: tokens 8+2t, 9+2t of head gi)
    const float pv0 = p[0] * vsc[0], pv1 = p[1] * vsc[0], pv2 = p[2] * vsc[1], pv3 = p[3] * vsc[1];
    const __half2 ht = __floats2half2_rn(pv0, pv1), hb = __floats2half2_rn(pv2, pv3);
    const float2 ft = __half22float2(ht), fb = __half22float2(hb);
    const uint32_t bh0 = movmatrix_trans(h2_as_u32(ht)), bh1 = movmatrix_trans(h2_as_u32(hb));
    const uint32_t bl0 = movmatrix_trans(h2_as_u32(__floats2half2_rn(pv0 - ft.x, pv1 - ft.y)));
    const uint32_t bl1 = movmatrix_trans(h2_as_u32(__floats2half2_rn(pv2 - fb.x, pv3 - fb.y)));
    // ---- V rows of tokens 2t, 2t+1, 8+2t, 9+2t (lane group gi's dims)
    uint32_t v0[NW], v1[NW], v8[NW], v9[NW];
    load_v_row<D, DT>(vd + (2 * t) * SG::kDb, vm + (2 * t) * SG::kMb, gi, v0);
    load_v_row<D, DT>(vd + (2 * t + 1) * SG::kDb, vm + (2 * t + 1) * SG::kMb, gi, v1);
    load_v_row<D, DT>(vd + (8 + 2 * t) * SG::kDb, vm + (8 + 2 * t) * SG::kMb, gi, v8);
    load_v_row<D, DT>(vd + (9 + 2 * t) * SG::kDb, vm + (9 + 2 * t) * SG::kMb, gi, v9);
    __syncwarp();
    // the slot is free: fetch the block kAttnSlots ahead into it
    if (j + kAttnSlots < nb) issue_block<D, DT>(slot, a.pool, a.layer, phys_of(j + kAttnSlots), gk, lane);
    cp_async_commit();
    slot_i = slot_i + 1 == kAttnSlots ? 0 : slot_i + 1;
    // A = V^T: row gi of m-tile m <- slot 2m, row gi+8 <- slot 2m+1; k-slots = tokens
#pragma unroll
    for (int m = 0; m < NV / 2; ++m) {
      const uint32_t a0 = pair_tokens(v0, v1, 2 * m), a1 = pair_tokens(v0, v1, 2 * m + 1);
      const uint32_t a2 = pair_tokens(v8, v9, 2 * m), a3 = pair_tokens(v8, v9, 2 * m + 1);
      mma_16816(acc[m], a0, a1, a2, a3, bh0, bh1);
      mma_16816(acc[m], a0, a1, a2, a3, bl0, bl1);
    }
  }
  cp_async_wait<0>();

  // ---- merge the NWARP warps of this block into the block's partial (m, l, o); the barrier below also
  // ends every warp's use of its ring, whose memory the merge reuses
  float l_tot[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float l = l_part[h];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    l_tot[h] = l;
  }
  if (gi == 0)
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (2 * t + h < G) {
        s_m[warp][2 * t + h] = m_run[h];
        s_l[warp][2 * t + h] = l_tot[h];
      }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int hd = 2 * t + h;
    if (hd >= G) continue;
    // this warp's share, rescaled to the block's running maximum of the head
    float mm = s_m[0][hd];
#pragma unroll
    for (int w = 1; w < NWARP; ++w) mm = fmaxf(mm, s_m[w][hd]);
    const float e = mm == -INFINITY ? 0.f : exp2f(m_run[h] - mm);
    float* dst = s_acc + (warp * 8 + hd) * D + gi * NV;
#pragma unroll
    for (int m = 0; m < NV / 2; ++m) {
      dst[v_slot_dim<DT>(2 * m)] = acc[m][h] * e;
      dst[v_slot_dim<DT>(2 * m + 1)] = acc[m][2 + h] * e;
    }
    if (warp == 0 && gi == 0) {
      float l = 0.f;
#pragma unroll
      for (int w = 0; w < NWARP; ++w) l += s_l[w][hd] * (mm == -INFINITY ? 0.f : exp2f(s_m[w][hd] - mm));
      s_pm[hd] = mm;  // -inf for a block without keys
      s_pl[hd] = l;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += blockDim.x) {
    const int h = idx / D, dim = idx - h * D;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) sum += s_acc[(w * 8 + h) * D + dim];
    s_po[idx] = sum;
  }
  if (threadIdx.x == 0) stamp(2);
  // ---- merge the cluster's splits through distributed shared memory: every rank stores its partials of
  // each rank's share of the outputs into that rank's inbox, then combines its own share from its inbox
  const int rank = (int)cluster.block_rank();
  const int per = (G * D + S - 1) / S;  // outputs of one rank's share
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  for (int idx = tid; idx < G * D; idx += blockDim.x) {
    const int r = idx / per;
    *cluster.map_shared_rank(&s_in_o[rank * per + (idx - r * per)], r) = s_po[idx];
  }
  if (tid < S * G) {
    const int r = tid / G, h = tid - r * G;
    *cluster.map_shared_rank(&s_in_m[rank][h], r) = s_pm[h];
    *cluster.map_shared_rank(&s_in_l[rank][h], r) = s_pl[h];
  }
  cluster.sync();  // release / acquire: every inbox is complete
  for (int idx = rank * per + tid; idx < min((rank + 1) * per, G * D); idx += blockDim.x) {
    const int h = idx / D, j = idx - rank * per;
    float mm = -INFINITY;
    for (int q = 0; q < S; ++q) mm = fmaxf(mm, s_in_m[q][h]);
    float l = 0.f, o = 0.f;
    for (int q = 0; q < S; ++q) {
      const float mq = s_in_m[q][h];
      const float e = mq == -INFINITY ? 0.f : exp2f(mq - mm);
      l = fmaf(s_in_l[q][h], e, l);
      o = fmaf(s_in_o[q * per + j], e, o);
    }
    if (K == 1) {
      a.o[(int64_t)b * a.ldo + (int64_t)gk * G * D + idx] = __float2half_rn(o / l);
    } else {  // this cluster's (m, l, o) of the output, for the merge of the K clusters
      float* pp = a.part + ((((int64_t)b * Hkv + gk) * kAttnMaxGroups + split / S) * 3) * G * D;
      pp[idx] = mm;  // -inf when none of the cluster's splits has a key
      pp[G * D + idx] = l;
      pp[2 * G * D + idx] = o;
    }
  }
  if (K > 1) {
    // the last block of the S K to arrive merges the K clusters' parts in cluster order (no waiting)
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const unsigned int n = atomicAdd(a.arrivals + (int64_t)b * Hkv + gk, 1u);
      s_last = n == (unsigned int)(S * K - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      const float* pb = a.part + (((int64_t)b * Hkv + gk) * kAttnMaxGroups) * 3 * G * D;
      merge_parts(pb, K, G * D, a.o + (int64_t)b * a.ldo + (int64_t)gk * G * D);
      if (tid == 0) a.arrivals[(int64_t)b * Hkv + gk] = 0u;  // ready for the next launch
    }
  }
  if (threadIdx.x == 0) stamp(3);
}

// ---------------------------------------------------------------- chunked prefill
// One block per (chunk token, KV head): its rotated k and v from the QKV output into the pool.
__global__ void kv_store_chunk_kernel(const KvChunkArgs a) {
  __shared__ __half xk[128], xv[128];
  __shared__ float red[8];
  const int t = blockIdx.x, h = blockIdx.y, i = threadIdx.x;
  const int d = a.pool.head_dim, Hkv = a.pool.n_kv_heads;
  pdl_wait();  // the QKV projection's output
  pdl_trigger();
  const __half* row = a.qkv + (int64_t)t * a.qkv_ld;
  xk[i] = row[(int64_t)(a.n_heads + h) * d + i];
  xv[i] = row[(int64_t)(a.n_heads + Hkv + h) * d + i];
  __syncthreads();
  const int pos = a.row_pos ? a.row_pos[t] : (a.step ? a.step->pos[0] : a.pos0) + t;
  const int sess = a.row_sess ? a.row_sess[t] : (a.step ? a.step->sess[0] : -1);
  const int32_t* table = sess >= 0 ? a.pool.tables + (int64_t)sess * a.pool.table_stride : a.table;
  const int blk = table[pos >> 4];
  if ((unsigned)blk >= (unsigned)a.pool.pool_blocks) {  // a table entry outside the pool: store nothing
    if (i == 0 && a.err) atomicOr(a.err, kErrBounds);
    return;
  }
  store_vec(a.pool, a.layer, blk, pos & 15, h, 0, xk, red);
  store_vec(a.pool, a.layer, blk, pos & 15, h, 1, xv, red);
}

// 8 consecutive values (dims c8 .. c8+7) of one pool vector in raw form: fp16 16 B, INT8 8 B + the
// vector's scale, INT4 4 B + the (scale, min) of their group.
struct RawUnit {
  uint4 d;
  uint32_t meta;
};
__device__ __forceinline__ RawUnit load_unit(const PoolGeom& P, int layer, int blk, int which, int head, int slot,
                                             int c8) {
  RawUnit r;
  r.meta = 0;
  const uint8_t* data = pool_vec(P, layer, blk, which, head, slot);
  if (P.kv_dtype == 0) {
    r.d = *reinterpret_cast<const uint4*>(data + c8 * 2);
  } else {
    const uint8_t* meta = pool_vec(P, layer, blk, which + 2, head, slot);
    if (P.kv_dtype == 1) {
      const uint2 v = *reinterpret_cast<const uint2*>(data + c8);
      r.d = make_uint4(v.x, v.y, 0, 0);
      r.meta = *reinterpret_cast<const uint16_t*>(meta);
    } else {
      r.d = make_uint4(*reinterpret_cast<const uint32_t*>(data + c8 / 2), 0, 0, 0);
      r.meta = reinterpret_cast<const uint32_t*>(meta)[c8 >> 5];
    }
  }
  return r;
}
// the unit as 8 fp16 values (INT8: s q; INT4: s q + m, in fp32 then rounded; FP16 as stored)
// the dequantised values of an INT8 / INT4 unit in fp32: s q (exact), s q + m (one rounding)
__device__ __forceinline__ void dequant_unit(int dt, const RawUnit& r, float (&v)[8]) {
  if (dt == 1) {
    const float s = __half2float(__ushort_as_half((unsigned short)r.meta));
    const int8_t* q = reinterpret_cast<const int8_t*>(&r.d);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = s * (float)q[e];
  } else {
    const __half2 sm = u32_as_h2(r.meta);
    const float s = __low2float(sm), mn = __high2float(sm);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __fadd_rn(__fmul_rn(s, (float)((r.d.x >> (4 * e)) & 15u)), mn);
  }
}
// the unit as 8 fp16 values (INT8 / INT4: the dequantised value rounded; FP16 as stored)
__device__ __forceinline__ void widen_unit(int dt, const RawUnit& r, __half (&h)[8]) {
  if (dt == 0) {
    *reinterpret_cast<uint4*>(h) = r.d;
    return;
  }
  float v[8];
  dequant_unit(dt, r, v);
#pragma unroll
  for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(v[e]);
}

// ---------------------------------------------------------------- prefill attention
// Block: one KV head and 4 warps x 16 MMA rows; a row is (token, query head of the group), 16/G tokens per
// warp. Keys go through shared memory in tiles of 64 (four pool blocks), K and V row-major as fp16 with
// padded rows, double-buffered: FP16 pools are copied with cp.async while the previous tile is computed,
// INT8 / INT4 pools are dequantised into the tile (s q, s q + m in fp32; keys as fp16 hi + lo, so QK^T sees
// the fp32 value, values rounded to fp16). Each warp runs QK^T
// (B fragments by ldmatrix), the causal mask, the online softmax and PV (B fragments by ldmatrix.trans,
// probabilities split into fp16 hi + lo) on m16n8k16 MMAs. Keys past the chunk's last token are zeros.
constexpr int kPfKeys = 64;  // keys per tile

template <int D>
struct PfGeom {
  static constexpr int kRow = D + 8;               // halves per shared-memory row (ldmatrix rows on distinct banks)
  static constexpr int kTile = kPfKeys * kRow;     // halves per K or V tile
  static constexpr size_t kBytes = (size_t)4 * kTile * 2;  // K and V, two buffers
  // INT8 / INT4 pools also keep the keys' low parts (k - fp16(k)), one tile per buffer after those
  static constexpr size_t kBytesQuant = (size_t)6 * kTile * 2;
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}

template <int D>
__global__ void __launch_bounds__(128) prefill_attn_kernel(const PrefillAttnArgs a) {
  using PG = PfGeom<D>;
  constexpr int KS = D / 16;  // k-steps of QK^T
  constexpr int NV = D / 8;   // n-tiles of PV
  constexpr int NT = kPfKeys / 8;  // n-tiles of QK^T per key tile
  extern __shared__ __align__(128) uint8_t smem[];
  __half* tiles = reinterpret_cast<__half*>(smem);  // [buf][K, V][kPfKeys][kRow]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int G = a.n_heads / a.n_kv_heads, gk = blockIdx.y;
  const int tpw = 16 / G;  // tokens per warp
  const int t_blk = blockIdx.x * 4 * tpw, t_warp = t_blk + warp * tpw;
  // this block's session: its rows of the QKV output and of o, its positions and block table
  const PfSeg sg = a.seg[blockIdx.z];
  if (t_blk >= sg.n_tok) return;  // past this session's tokens (grid.x covers the longest)
  const int n_tok = sg.n_tok, pos0 = sg.pos0;
  const int32_t* table = a.pool.tables + (int64_t)sg.sess * a.pool.table_stride;
  const __half* qkv = a.qkv + (int64_t)sg.row0 * a.qkv_ld;
  __half* o_rows = a.o + (int64_t)sg.row0 * a.ldo;
  const int dt = a.pool.kv_dtype;
  const int n_valid = pos0 + n_tok;  // keys in the pool after the chunk's store
  const int last_tok = min(n_tok, t_blk + 4 * tpw) - 1;
  const int n_keys = pos0 + last_tok + 1;  // keys this block reads
  const int n_tiles = (n_keys + kPfKeys - 1) / kPfKeys;
  const int warp_last = min(n_tok, t_warp + tpw) - 1;  // this warp's last token (may be < t_warp)

  // K data of (this layer, pool block 0, this KV head, slot 0); a block's V data is pool_v_off further
  const uint8_t* pool_head0 = pool_vec(a.pool, a.layer, 0, 0, gk, 0);
  const int64_t pool_v_off = pool_vec(a.pool, a.layer, 0, 1, gk, 0) - pool_head0;
  // key tile i into buffer bf: FP16 by cp.async (committed as one group), others widened synchronously.
  // Keys past the chunk's last stored token are zeros.
  auto stage = [&](int i, int bf) {
    __half* kt = tiles + (size_t)bf * 2 * PG::kTile;
    __half* vt = kt + PG::kTile;
    __half* klo = tiles + (size_t)(4 + bf) * PG::kTile;  // INT8 / INT4 only
    const int n_rows = max(0, min(kPfKeys, n_valid - i * kPfKeys));  // rows that exist in the pool
    if (dt == 0) {
      // a thread keeps one 16-byte column c8 of slots r0 + kRpp jj of every pool block of the tile (kRpp
      // rows per pass); only the block's base address changes from one pool block to the next
      constexpr int kCpr = D / 8, kRpp = 128 / kCpr;  // 16-byte chunks per row, rows per pass
      const int c8 = (tid % kCpr) * 8, r0 = tid / kCpr;
#pragma unroll
      for (int pb = 0; pb < 4; ++pb) {
        const int blk = i * 4 + pb;
        const int pbk = blk * 16 < n_valid ? checked_block(table[blk], a.pool.pool_blocks, a.err) : 0;
        const uint8_t* kb = pool_head0 + (int64_t)pbk * a.pool.block_bytes +
                            r0 * (2 * D) + c8 * 2;
#pragma unroll
        for (int jj = 0; jj < 16 / kRpp; ++jj) {
          const int row = pb * 16 + r0 + kRpp * jj;
          __half* dk = kt + row * PG::kRow + c8;
          __half* dv = vt + row * PG::kRow + c8;
          if (row < n_rows) {
            cp_async16(dk, kb + jj * kRpp * (2 * D));
            cp_async16(dv, kb + pool_v_off + jj * kRpp * (2 * D));
          } else {
            *reinterpret_cast<uint4*>(dk) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(dv) = make_uint4(0, 0, 0, 0);
          }
        }
      }
    } else {
      constexpr int kChunks = kPfKeys * D / 8;  // 16-byte chunks per K or V tile
      for (int c = tid; c < 2 * kChunks; c += 128) {
        const int which = c >= kChunks, cc = which ? c - kChunks : c;
        const int row = cc / (D / 8), c8 = (cc - row * (D / 8)) * 8;
        const int kp = i * kPfKeys + row;
        __half* dst = (which ? vt : kt) + row * PG::kRow + c8;
        __half* dlo = klo + row * PG::kRow + c8;  // keys only
        if (row >= n_rows) {
          *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
          if (!which) *reinterpret_cast<uint4*>(dlo) = make_uint4(0, 0, 0, 0);
          continue;
        }
        float v[8];
        dequant_unit(dt, load_unit(a.pool, a.layer, checked_block(table[kp >> 4], a.pool.pool_blocks, a.err), which, gk,
                                   kp & 15, c8),
                     v);
        __half h[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          h[e] = __float2half_rn(v[e]);
          lo[e] = __float2half_rn(v[e] - __half2float(h[e]));  // keys: hi + lo carries the fp32 value
        }
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<uint4*>(h);
        if (!which) *reinterpret_cast<uint4*>(dlo) = *reinterpret_cast<uint4*>(lo);
      }
    }
    cp_async_commit();
  };

  pdl_wait();
  pdl_trigger();
  // the rows of this lane: r0 = g, r1 = g + 8
  int tok[2], hq[2];
  bool live[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = g + 8 * h, tl = r / G;
    tok[h] = t_warp + tl;
    hq[h] = gk * G + (r - tl * G);
    live[h] = tl < tpw && tok[h] < n_tok;
  }
  if (n_tiles > 0) stage(0, 0);
  uint32_t qa[KS][4];
#pragma unroll
  for (int s = 0; s < KS; ++s)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half* q = qkv + (int64_t)(live[h] ? tok[h] : 0) * a.qkv_ld + (int64_t)hq[h] * D + 16 * s + 2 * t;
      qa[s][h] = live[h] ? *reinterpret_cast<const uint32_t*>(q) : 0u;
      qa[s][2 + h] = live[h] ? *reinterpret_cast<const uint32_t*>(q + 8) : 0u;
    }
  const float sc = 1.4426950408889634f / sqrtf((float)D);  // log2(e) / sqrt(d)
  float m_run[2] = {-1e30f, -1e30f}, l_run[2] = {0.f, 0.f};
  float acc[NV][4];
#pragma unroll
  for (int n = 0; n < NV; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

  for (int i = 0; i < n_tiles; ++i) {
    const int bf = i & 1;
    cp_async_wait<0>();
    __syncthreads();  // tile i is in; every warp is done with tile i - 1, whose buffer the next stage reuses
    if (i + 1 < n_tiles) stage(i + 1, bf ^ 1);
    const __half* kt = tiles + (size_t)bf * 2 * PG::kTile;
    const __half* vt = kt + PG::kTile;
    const __half* klo = tiles + (size_t)(4 + bf) * PG::kTile;
    if (warp_last < t_warp || i * kPfKeys > pos0 + warp_last) continue;  // no key of this tile is visible
    // ---- S = Q K^T over the tile's 64 keys: n-tile nt = keys 8 nt .. 8 nt + 7
    float sfr[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      sfr[nt][0] = sfr[nt][1] = sfr[nt][2] = sfr[nt][3] = 0.f;
#pragma unroll
      for (int s = 0; s < KS; s += 2) {
        // matrices: (k-step s, dims lo), (s, hi), (s + 1, lo), (s + 1, hi) of keys 8 nt ..
        const int m = lane >> 3;
        uint32_t kb[4];
        const int off = (8 * nt + (lane & 7)) * PG::kRow + 16 * (s + (m >> 1)) + 8 * (m & 1);
        ldsm_x4(kb, kt + off);
        mma_16816(sfr[nt], qa[s][0], qa[s][1], qa[s][2], qa[s][3], kb[0], kb[1]);
        mma_16816(sfr[nt], qa[s + 1][0], qa[s + 1][1], qa[s + 1][2], qa[s + 1][3], kb[2], kb[3]);
        if (dt != 0) {  // the keys' low parts
          ldsm_x4(kb, klo + off);
          mma_16816(sfr[nt], qa[s][0], qa[s][1], qa[s][2], qa[s][3], kb[0], kb[1]);
          mma_16816(sfr[nt], qa[s + 1][0], qa[s + 1][1], qa[s + 1][2], qa[s + 1][3], kb[2], kb[3]);
        }
      }
    }
    // causal mask and online softmax; fragment (nt, j): row g + 8 (j >> 1), key 64 i + 8 nt + 2 t + (j & 1)
    float mx[2] = {-1e30f, -1e30f};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int h = j >> 1, kp = i * kPfKeys + 8 * nt + 2 * t + (j & 1);
        const bool ok = live[h] && kp <= pos0 + tok[h];
        const float v = ok ? sfr[nt][j] * sc : -INFINITY;
        sfr[nt][j] = v;
        mx[h] = fmaxf(mx[h], v);
      }
    float corr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      const float mn = fmaxf(m_run[h], mx[h]);
      corr[h] = exp2f(m_run[h] - mn);
      m_run[h] = mn;
    }
    float ps[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int h = j >> 1;
        sfr[nt][j] = exp2f(sfr[nt][j] - m_run[h]);  // masked: exp2(-inf) = 0
        ps[h] += sfr[nt][j];
      }
#pragma unroll
    for (int h = 0; h < 2; ++h) l_run[h] = l_run[h] * corr[h] + ps[h];
#pragma unroll
    for (int n = 0; n < NV; ++n) {
      acc[n][0] *= corr[0];
      acc[n][1] *= corr[0];
      acc[n][2] *= corr[1];
      acc[n][3] *= corr[1];
    }
    // ---- O += P V, k-step j = keys 16 j .. 16 j + 15: P of n-tiles 2j, 2j+1 as the A operand, fp16 hi + lo
#pragma unroll
    for (int j = 0; j < NT / 2; ++j) {
      uint32_t ph[4], pl[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int nt = 2 * j + (q >> 1), h = q & 1;
        const float x0 = sfr[nt][2 * h], x1 = sfr[nt][2 * h + 1];
        const __half2 hh = __floats2half2_rn(x0, x1);
        const float2 hf = __half22float2(hh);
        ph[q] = h2_as_u32(hh);
        pl[q] = h2_as_u32(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
      }
#pragma unroll
      for (int n = 0; n < NV; n += 2) {
        // matrices: (dims 8n, keys lo), (8n, keys hi), (8n + 8, lo), (8n + 8, hi), transposed
        const int m = lane >> 3;
        uint32_t vb[4];
        ldsm_x4_t(vb, vt + (16 * j + 8 * (m & 1) + (lane & 7)) * PG::kRow + 8 * (n + (m >> 1)));
        mma_16816(acc[n], ph[0], ph[1], ph[2], ph[3], vb[0], vb[1]);
        mma_16816(acc[n], pl[0], pl[1], pl[2], pl[3], vb[0], vb[1]);
        mma_16816(acc[n + 1], ph[0], ph[1], ph[2], ph[3], vb[2], vb[3]);
        mma_16816(acc[n + 1], pl[0], pl[1], pl[2], pl[3], vb[2], vb[3]);
      }
    }
  }
  // normalise and store: acc[n][2h + j] = (row g + 8h, dim 8n + 2t + j)
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float l = l_run[h];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (!live[h]) continue;
    const float inv = l > 0.f ? 1.0f / l : 0.f;
    __half* o = o_rows + (int64_t)tok[h] * a.ldo + (int64_t)hq[h] * D;
#pragma unroll
    for (int n = 0; n < NV; ++n)
      *reinterpret_cast<__half2*>(o + 8 * n + 2 * t) = __floats2half2_rn(acc[n][2 * h] * inv, acc[n][2 * h + 1] * inv);
  }
}

template <typename K, typename Args>
cudaError_t launch_ex(const Launch& L, K kern, dim3 grid, dim3 block, size_t smem, const Args& a,
                      int cluster_x = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
  int n = 1;
  if (cluster_x > 0) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  if (L.counter) ++*L.counter;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int D, int DT, int NW>
cudaError_t attn_prepare() {
  auto kern = attn_kernel<D, DT, NW>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem_bytes<D, DT, NW>());
  if (e != cudaSuccess) return e;
  // the largest shared-memory carveout, as the GEMVs before and after use: an SM that switches carveouts
  // between kernels must drain and reconfigure before the next kernel's blocks can start on it
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int D, int DT, int NW>
cudaError_t launch_attn_nw(const Launch& L, const AttnArgs& a, int batch) {
  cudaError_t e = attn_prepare<D, DT, NW>();
  if (e != cudaSuccess) return e;
  return launch_ex(L, attn_kernel<D, DT, NW>, dim3(a.n_split * a.n_groups, a.n_kv_heads, batch), dim3(32 * NW),
                   attn_smem_bytes<D, DT, NW>(), a, a.n_split);
}

template <int D, int DT>
cudaError_t launch_attn_t(const Launch& L, const AttnArgs& a, int batch) {
  return a.wide ? launch_attn_nw<D, DT, attn_wide_warps<D, DT>()>(L, a, batch) : launch_attn_nw<D, DT, 4>(L, a, batch);
}

// Largest cluster size (16, 8, 4, 2, 1) of which at least one cluster fits on the device.
template <int D, int DT, int NW>
cudaError_t attn_max_cluster_nw(int* out) {
  cudaError_t e = attn_prepare<D, DT, NW>();
  if (e != cudaSuccess) return e;
  for (int s = 16; s >= 1; s /= 2) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(s, 1, 1);
    cfg.blockDim = dim3(32 * NW);
    cfg.dynamicSmemBytes = attn_smem_bytes<D, DT, NW>();
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = s;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, attn_kernel<D, DT, NW>, &cfg);
    if (e != cudaSuccess) return e;
    if (n >= 1) {
      *out = s;
      return cudaSuccess;
    }
  }
  *out = 0;
  return cudaErrorInvalidConfiguration;
}

}  // namespace

cudaError_t launch_kv_store(const Launch& L, const KvStoreArgs& a) {
  if (a.n_tok == 0) return cudaSuccess;
  return launch_ex(L, kv_store_kernel, dim3(a.n_tok, a.pool.n_kv_heads, a.n_layers), dim3(a.pool.head_dim), 0, a);
}

cudaError_t launch_kv_store_chunk(const Launch& L, const KvChunkArgs& a) {
  if (a.n_tok == 0) return cudaSuccess;
  return launch_ex(L, kv_store_chunk_kernel, dim3(a.n_tok, a.pool.n_kv_heads), dim3(a.pool.head_dim), 0, a);
}

cudaError_t launch_prefill_attention(const Launch& L, const PrefillAttnArgs& a) {
  if (a.n_seg < 1 || a.n_seg > MAG_MAX_BATCH) return cudaErrorInvalidValue;
  const int G = a.n_heads / a.n_kv_heads;
  if (G < 1 || G > 16) return cudaErrorInvalidValue;
  const int per_block = 4 * (16 / G);
  int longest = 0;
  for (int i = 0; i < a.n_seg; ++i) longest = a.seg[i].n_tok > longest ? a.seg[i].n_tok : longest;
  if (longest == 0) return cudaSuccess;
  const dim3 grid((longest + per_block - 1) / per_block, a.n_kv_heads, a.n_seg);
  auto run = [&](auto kern, size_t smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return e != cudaSuccess ? e : launch_ex(L, kern, grid, dim3(128), smem, a);
  };
  const bool quant = a.pool.kv_dtype != 0;
  if (a.head_dim == 128) return run(prefill_attn_kernel<128>, quant ? PfGeom<128>::kBytesQuant : PfGeom<128>::kBytes);
  if (a.head_dim == 64) return run(prefill_attn_kernel<64>, quant ? PfGeom<64>::kBytesQuant : PfGeom<64>::kBytes);
  return cudaErrorInvalidValue;
}

template <int D, int DT>
cudaError_t attn_max_cluster_t(int* out, bool wide) {
  return wide ? attn_max_cluster_nw<D, DT, attn_wide_warps<D, DT>()>(out) : attn_max_cluster_nw<D, DT, 4>(out);
}

cudaError_t attention_max_cluster(int head_dim, int kv_dtype, bool wide, int* out) {
  if (head_dim == 128) {
    if (kv_dtype == 0) return attn_max_cluster_t<128, 0>(out, wide);
    if (kv_dtype == 1) return attn_max_cluster_t<128, 1>(out, wide);
    return attn_max_cluster_t<128, 2>(out, wide);
  }
  if (head_dim == 64) {
    if (kv_dtype == 0) return attn_max_cluster_t<64, 0>(out, wide);
    if (kv_dtype == 1) return attn_max_cluster_t<64, 1>(out, wide);
    return attn_max_cluster_t<64, 2>(out, wide);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention(const Launch& L, const AttnArgs& a, int batch) {
  const int dt = a.pool.kv_dtype;
  if (a.n_split < 1 || a.n_split > 16 || a.n_groups < 1 || a.n_groups > kAttnMaxGroups ||
      (a.n_groups > 1 && (!a.part || !a.arrivals)))
    return cudaErrorInvalidValue;
  if (a.head_dim == 128) {
    if (dt == 0) return launch_attn_t<128, 0>(L, a, batch);
    if (dt == 1) return launch_attn_t<128, 1>(L, a, batch);
    return launch_attn_t<128, 2>(L, a, batch);
  }
  if (a.head_dim == 64) {
    if (dt == 0) return launch_attn_t<64, 0>(L, a, batch);
    if (dt == 1) return launch_attn_t<64, 1>(L, a, batch);
    return launch_attn_t<64, 2>(L, a, batch);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mag
