// fp16 matrix-vector product of the decode step above 4 tokens (the LM head) on mma.sync.
//
// logits[b][n] = sum_k W[n][k] xn[b][k], W the fp16 LM head in 2048-byte tiles
// (16 rows x 64 k, lane order: lane L's 64 bytes at 64 L), xn the final
// RMSNorm of the residual ("5. Core modules" 5.1, pre-norm). K-split grid: a
// block of 8 warps owns 8 x tpw tiles over a k-range whose activations fit in
// 64 KB of shared memory; warp w takes tiles mt0 + 8 i (i < tpw) one after
// the other through a per-warp ring of cp.async copies (16 bytes per lane, L2
// only) that runs on across them, filled before the programmatic-dependent-
// launch wait; m16n8k16 MMAs with fp32 accumulators, 8-token column tiles.
// The k-ranges of a tile are added in order by the last block of the column
// to arrive (a counter per block column), then one warp per tile writes it.
#include "kernels.h"
#include "gemv_epi.cuh"

namespace mag {

namespace {

constexpr int kWarps = 8;                  // warps per block
constexpr int kSlots = 4;                  // ring slots per warp
constexpr int kSlotBytes = 2048;           // one 16-row x 64-k fp16 tile

__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// copy chunk c of tile mt into a ring slot: each lane its 64 bytes
__device__ __forceinline__ void issue(uint8_t* slot, const GemvArgs& a, int mt, int c, int lane) {
  const uint8_t* src = a.w + ((int64_t)mt * a.n_chunks + c) * kSlotBytes + lane * 64;
  uint8_t* d = slot + lane * 64;
  cp_async16(d, src);
  cp_async16(d + 16, src + 16);
  cp_async16(d + 32, src + 32);
  cp_async16(d + 48, src + 48);
}

// Lane L's 64 bytes of a tile: rows g (g0, g1) and g+8 (h0, h1) at k = 16t .. 16t+15 of the chunk.
struct Stage {
  uint4 g0, g1, h0, h1;
};
__device__ __forceinline__ void read_slot(Stage& st, const uint8_t* slot, int lane) {
  const uint4* p = reinterpret_cast<const uint4*>(slot + lane * 64);
  st.g0 = p[0];
  st.g1 = p[1];
  st.h0 = p[2];
  st.h1 = p[3];
}

// Shared-memory staging of one block: B token rows of `xrow` halves (the block's k-range).
struct Staged {
  const __half* x;
  int xrow, c0;  // c0: first chunk of the staged range
};

template <int NT>
__device__ __forceinline__ void compute_chunk(const Stage& st, float (&acc)[2][4], const Staged& S, int B, int c,
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

// +8 halves per row: the rows of a quarter-warp's 16-byte loads fall on different banks
__host__ __device__ __forceinline__ size_t staged_bytes(int B, int nch) {
  return ((size_t)B * (nch * 64 + 8) * 2 + 127) & ~(size_t)127;
}

// Stage chunks [c0, c1) of xn = fp16(r / sqrt(mean(r^2) + eps) * gamma), the mean from the producer's n_ss
// partial sums of squares per token.
__device__ Staged stage_x(const GemvArgs& a, uint8_t* smem, float* s_inv, int c0, int c1) {
  const int tid = threadIdx.x, B = a.batch;
  Staged S;
  S.c0 = c0;
  S.xrow = (c1 - c0) * 64 + 8;
  __half* xw = reinterpret_cast<__half*>(smem);
  S.x = xw;
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
  const int units = (c1 - c0) * 8;
  for (int i = tid; i < B * units; i += blockDim.x) {
    const int b = i / units, u = i - b * units;
    const int k = (c0 * 8 + u) * 8;
    __half h[8];
    if (k >= a.K) {
#pragma unroll
      for (int e = 0; e < 8; ++e) h[e] = __float2half_rn(0.f);
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
    *reinterpret_cast<uint4*>(xw + (size_t)b * S.xrow + 8 * u) = *reinterpret_cast<const uint4*>(h);
  }
  __syncthreads();
  return S;
}

// Block: kWarps x TPW tiles over one k-range; warp w takes tiles mt0 + kWarps i (i < TPW) one after the
// other, its ring running on across them, so the block's activation staging serves TPW tiles per warp.
template <int NT, int TPW>
__global__ void __launch_bounds__(256) gemv_ksplit_kernel(const GemvArgs a) {
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
  uint8_t* ring = smem + staged_bytes(a.batch, a.chunks_per_cta) + (size_t)warp * kSlots * kSlotBytes;

#pragma unroll
  for (int u = 0; u < kSlots; ++u) {
    if (u < total) issue(ring + u * kSlotBytes, a, mt0 + kWarps * (u / n), c0 + u % n, lane);
    cp_async_commit();
  }

  pdl_wait();
  pdl_trigger();
  const Staged S = stage_x(a, smem, s_inv, c0, c1);

  float acc[2][4] = {};
  float accs[TPW][2][4];
  int si = 0, ti = 0, ci = 0;  // ring slot; tile and chunk of pair p
  // tile and chunk of the pair kSlots ahead (the next copy), advanced without divisions
  int qt = TPW == 1 ? 0 : kSlots / n, qc = TPW == 1 ? kSlots : kSlots - qt * n;
  for (int p = 0; p < total; ++p) {
    uint8_t* slot = ring + si * kSlotBytes;
    if (++si == kSlots) si = 0;
    cp_async_wait<kSlots - 1>();
    __syncwarp();
    Stage cur;
    read_slot(cur, slot, lane);
    __syncwarp();
    if (p + kSlots < total) issue(slot, a, mt0 + kWarps * qt, c0 + qc, lane);
    cp_async_commit();
    if (TPW > 1 && ++qc == n) {
      qc = 0;
      ++qt;
    } else if (TPW == 1) {
      ++qc;
    }
    compute_chunk<NT>(cur, acc, S, a.batch, c0 + (TPW == 1 ? p : ci), g, t);
    if (TPW > 1 && ++ci == n) {  // tile ti complete
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
        for (int j = 0; j < 4; ++j) acc[nt][j] = 0.f;
      ci = 0;
      ++ti;
    }
  }
  if (TPW == 1 && nv)  // one tile: its result once the loop is done
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) accs[0][nt][j] = acc[nt][j];
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
    tokepi::epilogue_tile<NT, EPI_STORE_OUT>(a, mt0 + kWarps * i, accs[i], lane);
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

cudaError_t launch_sched(const Launch& L, const GemvArgs& a) {
  const size_t smem = gemv_smem_bytes(a, W_F16);
  const int tpw = a.tpw == 4 ? 4 : (a.tpw == 2 ? 2 : 1);
  const dim3 grid((a.n_mtiles + kWarps * tpw - 1) / (kWarps * tpw), a.ks);
  if (a.batch > 8) {
    if (tpw == 4) return launch_k(L, gemv_ksplit_kernel<2, 4>, grid, smem, a);
    if (tpw == 2) return launch_k(L, gemv_ksplit_kernel<2, 2>, grid, smem, a);
    return launch_k(L, gemv_ksplit_kernel<2, 1>, grid, smem, a);
  }
  if (tpw == 4) return launch_k(L, gemv_ksplit_kernel<1, 4>, grid, smem, a);
  if (tpw == 2) return launch_k(L, gemv_ksplit_kernel<1, 2>, grid, smem, a);
  return launch_k(L, gemv_ksplit_kernel<1, 1>, grid, smem, a);
}

}  // namespace

size_t gemv_smem_bytes(const GemvArgs& a, int wfmt) {
  (void)wfmt;
  return staged_bytes(a.batch, a.chunks_per_cta) + (size_t)kWarps * kSlots * kSlotBytes;
}

cudaError_t launch_gemv(const Launch& L, const GemvArgs& a, int wfmt, int xsrc, int epi) {
  if (a.batch <= kPipeMaxBatch) return launch_gemv_pipe(L, a, wfmt, xsrc, epi);
  if (wfmt == W_W4) return launch_gemv_batch(L, a, xsrc, epi);
  if (wfmt == W_F16 && xsrc == XSRC_RESID && epi == EPI_STORE_OUT) return launch_sched(L, a);
  return cudaErrorInvalidValue;
}

}  // namespace mag
