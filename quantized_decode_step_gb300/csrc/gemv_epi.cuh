// Per-tile epilogue of the decode GEMVs above 4 tokens (k_gemv.cu, k_gemv_batch.cu): one warp writes the
// 16 rows x up to 16 tokens of a finished tile.
#pragma once
#include "kernels.h"

namespace mag {
namespace tokepi {

__device__ __forceinline__ float silu_mul(float gte, float up) { return gte / (1.0f + expf(-gte)) * up; }

// Per-tile epilogue, one warp. acc[nt][0..1]: row g, tokens 8nt+2t, +1; acc[nt][2..3]: row g+8.
template <int NT, int EPI>
__device__ __forceinline__ void epilogue_tile(const GemvArgs& a, int mt, const float (&acc)[2][4], int lane) {
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

}  // namespace tokepi
}  // namespace mag
