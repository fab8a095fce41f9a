// W4A16 (and fp16) matrix-vector products of the decode step on mma.sync.
//
// y[b][n] = sum_k deq(W)[n][k] x[b][k] for a handful of tokens b, with the
// weights streamed once from HBM ("5. Core modules" 5.1: 4-bit weights, FP16
// activations). At load time each projection is repacked into 640-byte tiles
// (16 rows x 64 k: 512 bytes of codes in lane order, then 128 bytes of fp16
// (scale, min) pairs), so a warp's per-chunk loads are two fully coalesced
// 128-bit loads per lane. A lane turns its 8-nibble words into exact small
// integers in fp16 with a LOP3 into the mantissa of 1024 (the int4-to-fp16
// conversion of Kim et al., "Who Says Elephants Can't Run", 2022) and feeds
// m16n8k16 tensor-core MMAs with fp32 accumulators, one fresh accumulator per
// 32-wide group; scale and min are applied per group in fp32:
//     sum_k (s q_k + m) x_k = s * sum_k q_k x_k + m * X_g,   X_g = sum_{k in g} x_k,
// so the product carries no rounding of the dequantised weights.
//
// The activations are staged once per block in shared memory, in 8-wide
// units ordered (x0,x4,x1,x5,x2,x6,x3,x7) -- the k order the nibble pairs come
// out in -- together with their group sums X_g. For the projections that
// follow an RMSNorm ("5. Core modules" 5.1, pre-norm) the staging computes the
// norm itself from the fp32 residual and the producer's per-tile sums of
// squares.
//
// Schedules:
//   Stream-K (up to 4 tokens): the (tile, chunk) pairs of the whole matrix are
//   cut into equal contiguous runs, one per warp of a grid sized to the GPU; a
//   tile split between warps is finished by the last of them to arrive, which
//   adds the parts in warp order (deterministic).
//   K-split (more tokens): a block owns 8 tiles over a k-range whose
//   activations fit in shared memory; k-ranges are merged in order by the last
//   block of the group.
// Epilogues (per tile, one warp): QKV (fp16, q and k rotated by the
// pre-generated RoPE table; the tile's rows g and g+8 are the pair (i, i+d/2)
// of one head), RESID (fp32 residual add + per-tile sums of squares), SWIGLU
// (silu(gate) * up of interleaved gate/up rows), OUT (fp16 logits into the
// caller's buffer).
//
// Weights reach shared memory through a per-warp ring of cp.async copies
// (16 bytes per lane, L2 only), 12 chunks deep for W4 tiles and 4 for fp16
// rows, so a warp keeps ~8 KB of HBM reads in flight without holding them in
// registers; the ring is filled before the programmatic-dependent-launch wait,
// so the first reads overlap the previous kernel.
#include "kernels.h"

namespace mag {

namespace {

constexpr int kWarps = 8;  // warps per block

__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Per-warp ring of weight chunks in shared memory.
template <int WFMT>
struct Ring;

template <>
struct Ring<W_W4> {
  static constexpr int kSlots = 12;
  static constexpr int kSlotBytes = kTileBytes;  // 512 B codes (lane order) + 128 B (scale, min)
  // copy chunk (mt, c) into `slot`: every lane its 16 B of codes, lanes 0-7 the (scale, min) rows
  static __device__ __forceinline__ void issue(uint8_t* slot, const GemvArgs& a, int mt, int c, int lane) {
    const uint8_t* tile = a.w + ((int64_t)mt * a.n_chunks + c) * kTileBytes;
    cp_async16(slot + lane * 16, tile + lane * 16);
    if (lane < 8) cp_async16(slot + 512 + lane * 16, tile + 512 + lane * 16);
  }
};

template <>
struct Ring<W_F16> {
  static constexpr int kSlots = 4;
  static constexpr int kSlotBytes = 2048;  // 16 rows x 64 k fp16 tile, lane order: lane L's 64 B at 64 L
  static __device__ __forceinline__ void issue(uint8_t* slot, const GemvArgs& a, int mt, int c, int lane) {
    const uint8_t* src = a.w + ((int64_t)mt * a.n_chunks + c) * kSlotBytes + lane * 64;
    uint8_t* d = slot + lane * 64;
    cp_async16(d, src);
    cp_async16(d + 16, src + 16);
    cp_async16(d + 32, src + 32);
    cp_async16(d + 48, src + 48);
  }
};

struct W4Stage {
  uint4 code;  // row g: group 0 word t, group 1 word t; row g+8: the same
  uint4 sm;    // (scale, min): row g group 0, group 1; row g+8 group 0, group 1
};
struct F16Stage {
  uint4 g0, g1, h0, h1;
};
__device__ __forceinline__ void read_slot(W4Stage& st, const uint8_t* slot, int lane) {
  st.code = *reinterpret_cast<const uint4*>(slot + lane * 16);
  st.sm = *reinterpret_cast<const uint4*>(slot + 512 + (lane >> 2) * 16);
}
__device__ __forceinline__ void read_slot(F16Stage& st, const uint8_t* slot, int lane) {
  const uint4* p = reinterpret_cast<const uint4*>(slot + lane * 64);
  st.g0 = p[0];
  st.g1 = p[1];
  st.h0 = p[2];
  st.h1 = p[3];
}
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

// The 8 codes of a word (k0 in bits 0-3 ... k7 in bits 28-31) as exact fp16
// values code * 2^-20, paired (k0,k4) (k1,k5) (k2,k6) (k3,k7): each pair is the
// word masked so that its two nibbles land in bits 4-7 and 20-23, i.e. in the
// mantissa of an fp16 subnormal (16 * code <= 240 units of 2^-24). Integer
// shifts and masks only; the tensor cores take the subnormals as they are.
struct Q4 {
  uint32_t e0, e1, e2, e3;
};
__device__ __forceinline__ Q4 codes_word(uint32_t w) {
  Q4 q;
  q.e0 = (w << 4) & 0x00F000F0u;
  q.e1 = w & 0x00F000F0u;
  q.e2 = (w >> 4) & 0x00F000F0u;
  q.e3 = (w >> 8) & 0x00F000F0u;
  return q;
}
constexpr float kCodeUnit = 1048576.0f;  // 2^20: undoes the code scaling of codes_word

// Shared-memory staging of one block: B token rows of `xrow` halves (the
// block's k-range in W4 unit order or natural order) followed by the group
// sums [B][grow] (W4 only).
struct Staged {
  const __half* x;
  const float* xs;
  int xrow, grow, c0;  // c0: first chunk of the staged range
};

// Per lane and n-tile: acc[0..3] collects scale * (codes . x) (in units of
// 2^-20) and acc[4..7] min * X_g, for (row g, token 2t), (row g, 2t+1),
// (row g+8, 2t), (row g+8, 2t+1).
template <int NT>
__device__ __forceinline__ void compute_chunk(const W4Stage& st, float (&acc)[2][8], const Staged& S, int B, int c,
                                              int g, int t) {
  const int cl = c - S.c0;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    // columns past the batch read a valid row and are discarded
    const int tok = min(g + 8 * nt, B - 1);
    const int t0 = min(8 * nt + 2 * t, B - 1), t1 = min(8 * nt + 2 * t + 1, B - 1);
    const uint4* xr = reinterpret_cast<const uint4*>(S.x + (size_t)tok * S.xrow) + 8 * cl + t;
    const float2 X0 = reinterpret_cast<const float2*>(S.xs + (size_t)t0 * S.grow)[cl];
    const float2 X1 = reinterpret_cast<const float2*>(S.xs + (size_t)t1 * S.grow)[cl];
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
      const Q4 qg = codes_word(grp ? st.code.y : st.code.x);
      const Q4 qv = codes_word(grp ? st.code.w : st.code.z);
      const uint4 xb = xr[4 * grp];
      float aq[4] = {0.f, 0.f, 0.f, 0.f};
      mma_16816(aq, qg.e0, qv.e0, qg.e1, qv.e1, xb.x, xb.y);
      mma_16816(aq, qg.e2, qv.e2, qg.e3, qv.e3, xb.z, xb.w);
      const float2 fg = __half22float2(u32_as_h2(grp ? st.sm.y : st.sm.x));
      const float2 fv = __half22float2(u32_as_h2(grp ? st.sm.w : st.sm.z));
      const float xs0 = grp ? X0.y : X0.x, xs1 = grp ? X1.y : X1.x;
      acc[nt][0] = fmaf(fg.x, aq[0], acc[nt][0]);
      acc[nt][4] = fmaf(fg.y, xs0, acc[nt][4]);
      acc[nt][2] = fmaf(fv.x, aq[2], acc[nt][2]);
      acc[nt][6] = fmaf(fv.y, xs0, acc[nt][6]);
      if (B > 1) {
        acc[nt][1] = fmaf(fg.x, aq[1], acc[nt][1]);
        acc[nt][5] = fmaf(fg.y, xs1, acc[nt][5]);
        acc[nt][3] = fmaf(fv.x, aq[3], acc[nt][3]);
        acc[nt][7] = fmaf(fv.y, xs1, acc[nt][7]);
      }
    }
  }
}

// The four results of an n-tile: W4 parts combined (2^20 undoes the code scaling).
__device__ __forceinline__ void tile_result(const float (&a)[8], float (&r)[4], int wfmt) {
#pragma unroll
  for (int i = 0; i < 4; ++i) r[i] = wfmt == W_W4 ? fmaf(a[i], kCodeUnit, a[i + 4]) : a[i];
}

template <int NT>
__device__ __forceinline__ void compute_chunk(const F16Stage& st, float (&acc)[2][8], const Staged& S, int B, int c,
                                              int g, int t) {
  const int cl = c - S.c0;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tok = min(g + 8 * nt, B - 1);  // columns past the batch read a valid row and are discarded
    const uint4* p = reinterpret_cast<const uint4*>(S.x + (size_t)tok * S.xrow);
    const uint4 x0 = p[8 * cl + 2 * t], x1 = p[8 * cl + 2 * t + 1];
    mma_16816(acc[nt], st.g0.x, st.h0.x, st.g0.y, st.h0.y, x0.x, x0.y);
    mma_16816(acc[nt], st.g0.z, st.h0.z, st.g0.w, st.h0.w, x0.z, x0.w);
    mma_16816(acc[nt], st.g1.x, st.h1.x, st.g1.y, st.h1.y, x1.x, x1.y);
    mma_16816(acc[nt], st.g1.z, st.h1.z, st.g1.w, st.h1.w, x1.z, x1.w);
  }
}

// position of element e (0..7) of a unit in the W4 activation order
__device__ __forceinline__ int unit_pos(int e) { return e < 4 ? 2 * e : 2 * (e - 4) + 1; }

// Stage chunks [c0, c1) of the activations into shared memory (and their group
// sums for W4). XSRC_RESID: xn = fp16(r / sqrt(mean(r^2) + eps) * gamma), the
// mean from the producer's n_ss partial sums of squares per token.
__host__ __device__ __forceinline__ size_t staged_bytes(int B, int nch) {
  return ((((size_t)B * (nch * 64 + 8) * 2 + 15) & ~(size_t)15) + (size_t)B * (2 * nch + 2) * 4 + 127) &
         ~(size_t)127;
}

template <int WFMT, int XSRC>
__device__ Staged stage_x(const GemvArgs& a, uint8_t* smem, float* s_inv, int c0, int c1) {
  const int tid = threadIdx.x, B = a.batch;
  Staged S;
  S.c0 = c0;
  S.xrow = (c1 - c0) * 64 + 8;
  S.grow = 2 * (c1 - c0) + 2;
  __half* xw = reinterpret_cast<__half*>(smem);
  float* xsw = reinterpret_cast<float*>(smem + (((size_t)B * S.xrow * 2 + 15) & ~(size_t)15));
  S.x = xw;
  S.xs = xsw;
  if (XSRC == XSRC_RESID) {
    // inv[b] from the producer's partial sums of squares (all threads share the loads)
    float part[MAG_MAX_BATCH];
    for (int b = 0; b < B; ++b) part[b] = 0.f;
    for (int i = tid; i < a.n_ss; i += blockDim.x)
      for (int b = 0; b < B; ++b) part[b] += __ldcg(a.ss_part + (int64_t)i * MAG_MAX_BATCH + b);
    for (int b = 0; b < B; ++b) {
      const float v = warp_sum(part[b]);
      if ((tid & 31) == 0) s_inv[(tid >> 5) * MAG_MAX_BATCH + b] = v;
    }
    __syncthreads();
    if (tid < B) {
      float tot = 0.f;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_inv[w * MAG_MAX_BATCH + tid];
      s_inv[kWarps * MAG_MAX_BATCH + tid] = 1.0f / sqrtf(tot / (float)a.K + a.eps);
    }
    __syncthreads();
  }
  const int units = (c1 - c0) * 8;  // multiple of 4: the 4 units of a group sit in one quad of lanes
  for (int base = 0; base < B * units; base += blockDim.x) {
    const int i = base + tid;
    const bool live = i < B * units;
    const int b = live ? i / units : 0, u = live ? i - b * units : 0;
    const int k = (c0 * 8 + u) * 8;
    float s = 0.f;
    if (live) {
      __half h[8];
      if (k >= a.K) {
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(0.f);
      } else if (XSRC == XSRC_F16) {
        *reinterpret_cast<uint4*>(h) = *reinterpret_cast<const uint4*>(a.x + (int64_t)b * a.ldx + k);
      } else {
        const float inv = s_inv[kWarps * MAG_MAX_BATCH + b];
        const float4 r0 = __ldcg(reinterpret_cast<const float4*>(a.r + (int64_t)b * a.ldr + k));
        const float4 r1 = __ldcg(reinterpret_cast<const float4*>(a.r + (int64_t)b * a.ldr + k + 4));
        const uint4 gg = *reinterpret_cast<const uint4*>(a.gamma + k);
        const __half* gh = reinterpret_cast<const __half*>(&gg);
        const float f[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(f[e] * inv * __half2float(gh[e]));
      }
      __half o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        o[WFMT == W_W4 ? unit_pos(e) : e] = h[e];
        s += __half2float(h[e]);
      }
      *reinterpret_cast<uint4*>(xw + (size_t)b * S.xrow + 8 * u) = *reinterpret_cast<uint4*>(o);
    }
    if (WFMT == W_W4) {
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (live && (u & 3) == 0) xsw[(size_t)b * S.grow + u / 4] = s;
    }
  }
  __syncthreads();
  return S;
}

__device__ __forceinline__ float silu_mul(float gte, float up) { return gte / (1.0f + expf(-gte)) * up; }

// Per-tile epilogue, one warp. acc[nt][0..1]: row g, tokens 8nt+2t, +1; acc[nt][2..3]: row g+8.
template <int NT, int EPI>
__device__ void epilogue_tile(const GemvArgs& a, int mt, const float (&acc)[2][4], int lane) {
  const int g = lane >> 2, t = lane & 3, B = a.batch;
  if (EPI == EPI_RESID) {
    float ssq[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
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
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        float v = ssq[nt][jj];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        const int tok = nt * 8 + 2 * t + jj;
        if (g == 0 && tok < B) a.ss_part[(int64_t)mt * MAG_MAX_BATCH + tok] = v;
      }
    return;
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int tok = nt * 8 + 2 * t + jj;
      if (tok >= B) continue;
      const float lo = acc[nt][jj], hi = acc[nt][jj + 2];  // rows g and g + 8 of the tile
      if (EPI == EPI_SWIGLU) {
        a.out_h[(int64_t)tok * a.ldo + mt * 8 + g] = __float2half_rn(silu_mul(lo, hi));
      } else if (EPI == EPI_QKV) {
        const int tiles_per_head = a.head_dim / 16, head = mt / tiles_per_head;
        const int i = 8 * (mt - head * tiles_per_head) + g;  // pair (i, i + d/2) of the head
        const int row = head * a.head_dim + i, row8 = row + a.head_dim / 2;
        __half* o = a.out_h + (int64_t)tok * a.ldo;
        if (head < a.n_rot_heads) {
          // round as the fp16 projection output, then rotate
          const float x0 = __half2float(__float2half_rn(lo)), x1 = __half2float(__float2half_rn(hi));
          const int pos = a.step->pos[tok], hd = a.head_dim / 2;
          const float cs = a.rope_cos[(int64_t)pos * hd + i], sn = a.rope_sin[(int64_t)pos * hd + i];
          o[row] = __float2half_rn(x0 * cs - x1 * sn);
          o[row8] = __float2half_rn(x0 * sn + x1 * cs);
        } else {
          o[row] = __float2half_rn(lo);
          o[row8] = __float2half_rn(hi);
        }
      } else {
        __half* o = reinterpret_cast<__half*>(a.step->out) + (int64_t)tok * a.ldo + mt * 16 + g;
        o[0] = __float2half_rn(lo);
        o[8] = __float2half_rn(hi);
      }
    }
}

// ------------------------------------------------------------------ K-split schedule (B > 4)
// Block: kWarps x TPW tiles over one k-range; warp w takes tiles mt0 + kWarps i (i < TPW) one after the
// other, its ring running on across them, so the block's activation staging serves TPW tiles per warp.
template <int NT, int TPW, int WFMT, int XSRC, int EPI>
__global__ void __launch_bounds__(256) gemv_ksplit_kernel(const GemvArgs a) {
  using Stage = typename StageT<WFMT>::type;
  using R = Ring<WFMT>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_inv[(kWarps + 1) * MAG_MAX_BATCH];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int mt0 = blockIdx.x * kWarps * TPW + warp;
  int nv = 0;  // this warp's tiles that exist (a prefix of its TPW)
#pragma unroll
  for (int i = 0; i < TPW; ++i) nv += mt0 + kWarps * i < a.n_mtiles;
  const int c0 = blockIdx.y * a.chunks_per_cta, c1 = min(c0 + a.chunks_per_cta, a.n_chunks);
  const int n = c1 - c0;        // chunks per tile
  const int total = nv * n;     // (tile, chunk) pairs of this warp, tile-major
  uint8_t* ring = smem + staged_bytes(a.batch, a.chunks_per_cta) + (size_t)warp * R::kSlots * R::kSlotBytes;

#pragma unroll
  for (int u = 0; u < R::kSlots; ++u) {
    if (u < total) R::issue(ring + u * R::kSlotBytes, a, mt0 + kWarps * (u / n), c0 + u % n, lane);
    cp_async_commit();
  }

  pdl_wait();
  pdl_trigger();
  const Staged S = stage_x<WFMT, XSRC>(a, smem, s_inv, c0, c1);

  float acc8[2][8] = {};
  float accs[TPW][2][4];
  int si = 0, ti = 0, ci = 0;  // ring slot; tile and chunk of pair p
  // tile and chunk of the pair kSlots ahead (the next copy), advanced without divisions
  int qt = TPW == 1 ? 0 : R::kSlots / n, qc = TPW == 1 ? R::kSlots : R::kSlots - qt * n;
  for (int p = 0; p < total; ++p) {
    uint8_t* slot = ring + si * R::kSlotBytes;
    if (++si == R::kSlots) si = 0;
    cp_async_wait<R::kSlots - 1>();
    __syncwarp();
    Stage cur;
    read_slot(cur, slot, lane);
    __syncwarp();
    if (p + R::kSlots < total) R::issue(slot, a, mt0 + kWarps * qt, c0 + qc, lane);
    cp_async_commit();
    if (TPW > 1 && ++qc == n) {
      qc = 0;
      ++qt;
    } else if (TPW == 1) {
      ++qc;
    }
    compute_chunk<NT>(cur, acc8, S, a.batch, c0 + (TPW == 1 ? p : ci), g, t);
    if (TPW > 1 && ++ci == n) {  // tile ti complete
      float acc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) tile_result(acc8[nt], acc[nt], WFMT);
#pragma unroll
      for (int i = 0; i < TPW; ++i)
        if (i == ti)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) accs[i][nt][j] = acc[nt][j];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc8[nt][j] = 0.f;
      ci = 0;
      ++ti;
    }
  }
  if (TPW == 1 && nv) {  // one tile: its result once the loop is done
    float acc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) tile_result(acc8[nt], acc[nt], WFMT);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) accs[0][nt][j] = acc[nt][j];
  }
  cp_async_wait<0>();
  if (a.ks > 1) {
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      if (i >= nv) break;
      const int mt = mt0 + kWarps * i;
      float* p = a.partial + (((size_t)blockIdx.y * a.n_mtiles + mt) * 32 + lane) * (4 * NT);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float4*>(p + nt * 4) =
            make_float4(accs[i][nt][0], accs[i][nt][1], accs[i][nt][2], accs[i][nt][3]);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(a.counters + blockIdx.x, 1u) == (unsigned)(a.ks - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
      if (i >= nv) break;
      const int mt = mt0 + kWarps * i;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) accs[i][nt][j] = 0.f;
      for (int s = 0; s < a.ks; ++s) {
        const float* p = a.partial + (((size_t)s * a.n_mtiles + mt) * 32 + lane) * (4 * NT);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(p + nt * 4));
          accs[i][nt][0] += v.x;
          accs[i][nt][1] += v.y;
          accs[i][nt][2] += v.z;
          accs[i][nt][3] += v.w;
        }
      }
    }
    if (tid == 0) a.counters[blockIdx.x] = 0;
  }
#pragma unroll
  for (int i = 0; i < TPW; ++i) {
    if (i >= nv) break;
    epilogue_tile<NT, EPI>(a, mt0 + kWarps * i, accs[i], lane);
  }
}

template <typename K>
cudaError_t launch_k(const Launch& L, K kern, dim3 grid, size_t smem, const GemvArgs& a) {
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(32 * kWarps);
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

template <int WFMT, int XSRC, int EPI>
cudaError_t launch_sched(const Launch& L, const GemvArgs& a) {
  const size_t smem = gemv_smem_bytes(a, WFMT);
  const int tpw = a.tpw == 4 ? 4 : (a.tpw == 2 ? 2 : 1);
  const dim3 grid((a.n_mtiles + kWarps * tpw - 1) / (kWarps * tpw), a.ks);
  if (a.batch > 8) {
    if (tpw == 4) return launch_k(L, gemv_ksplit_kernel<2, 4, WFMT, XSRC, EPI>, grid, smem, a);
    if (tpw == 2) return launch_k(L, gemv_ksplit_kernel<2, 2, WFMT, XSRC, EPI>, grid, smem, a);
    return launch_k(L, gemv_ksplit_kernel<2, 1, WFMT, XSRC, EPI>, grid, smem, a);
  }
  if (tpw == 4) return launch_k(L, gemv_ksplit_kernel<1, 4, WFMT, XSRC, EPI>, grid, smem, a);
  if (tpw == 2) return launch_k(L, gemv_ksplit_kernel<1, 2, WFMT, XSRC, EPI>, grid, smem, a);
  return launch_k(L, gemv_ksplit_kernel<1, 1, WFMT, XSRC, EPI>, grid, smem, a);
}

}  // namespace

size_t gemv_smem_bytes(const GemvArgs& a, int wfmt) {
  const int nch = a.chunks_per_cta;
  const size_t ring = wfmt == W_W4 ? (size_t)Ring<W_W4>::kSlots * Ring<W_W4>::kSlotBytes
                                   : (size_t)Ring<W_F16>::kSlots * Ring<W_F16>::kSlotBytes;
  return staged_bytes(a.batch, nch) + kWarps * ring;
}

cudaError_t launch_gemv(const Launch& L, const GemvArgs& a, int wfmt, int xsrc, int epi) {
  if (a.n_cta > 0) return launch_gemv_pipe(L, a, wfmt, xsrc, epi);
#define MAG_GEMV_CASE(W_, X_, E_) \
  if (wfmt == W_ && xsrc == X_ && epi == E_) return launch_sched<W_, X_, E_>(L, a);
  MAG_GEMV_CASE(W_W4, XSRC_RESID, EPI_QKV)
  MAG_GEMV_CASE(W_W4, XSRC_F16, EPI_RESID)
  MAG_GEMV_CASE(W_W4, XSRC_RESID, EPI_SWIGLU)
  MAG_GEMV_CASE(W_F16, XSRC_RESID, EPI_STORE_OUT)
#undef MAG_GEMV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace mag
