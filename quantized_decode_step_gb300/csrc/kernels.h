// Host-side launch interfaces of the decode-step kernels.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace mag {

// Launch helper: every kernel goes through cudaLaunchKernelEx so that the
// programmatic-dependent-launch attribute can be set uniformly.
struct Launch {
  cudaStream_t stream;
  bool pdl;
  int* counter;  // incremented per launch (may be null)
};

// ---------------------------------------------------------------- W4 / fp16 GEMV (mma.sync)
enum WeightFmt { W_W4 = 0, W_F16 = 1 };
enum XMode { X_DIRECT = 0, X_SMEM = 1 };
enum Epilogue { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_STORE_OUT = 3 };
enum Tail { TAIL_NONE = 0, TAIL_NORM = 1, TAIL_HIDDEN = 2 };

struct GemvArgs {
  const uint8_t* w;       // W4 codes [N][w_row_bytes] or fp16 [N][K]
  const __half2* sm;      // W4 (scale, min) pairs [N][sm_row]
  int64_t w_row_bytes;
  int32_t sm_row;         // groups per row (W4)
  int32_t n_mtiles;       // 16-row tiles (SwiGLU: 8 gate + 8 up rows; QKV: rows i..i+7 and i+d/2.. of a head)
  int32_t K;              // reduction length
  int32_t n_chunks;       // ceil(K / 64)
  int32_t chunks_per_cta; // k-range of one block, in 64-wide chunks
  int32_t ks;             // k-splits (grid.y)
  int32_t mpc;            // m-tiles per block
  int32_t wk;             // warps sharing one m-tile's k-range
  const __half* x;        // activations [B][ldx]: W4 unit order (x0,x4,x1,x5,x2,x6,x3,x7) / natural (fp16 W)
  int32_t ldx;
  const float* xsum;      // W4: group sums of x [B][ldxs]
  int32_t ldxs;
  int32_t batch;
  // EPI_QKV
  int32_t head_dim, n_rot_heads;
  const float* rope_cos;
  const float* rope_sin;
  // EPI_QKV / EPI_SWIGLU: fp16 out [B][ldo]; EPI_SWIGLU group sums [B][ldos]
  __half* out_h;
  int32_t ldo;
  int32_t swiglu_f;
  float* out_sum;
  int32_t ldos;
  // EPI_RESID: residual [B][ldr] += y, per-tile sums of squares [n_mtiles][16], tail
  float* r;
  int32_t ldr;
  float* ss_part;
  int32_t tail;           // Tail
  const __half* gamma;    // TAIL_NORM gain
  float eps;
  __half* xn;             // TAIL_NORM output [B][ldxn]
  int32_t ldxn;
  int32_t xn_permuted;    // 1: W4 unit order
  float* xn_sum;          // group sums of xn (or null) [B][ldxns]
  int32_t ldxns;
  float* partial;         // ks > 1: [ks][n_mtiles][32][4 * n_tiles]
  uint32_t* counters;     // [grid.x + 1], zero between launches
  const StepArgs* step;
};

size_t gemv_smem_bytes(const GemvArgs& a, int xmode);
cudaError_t launch_gemv(const Launch& L, const GemvArgs& a, int wfmt, int xmode, int epi);

// ---------------------------------------------------------------- step prologue
// block-table writes, fp16 input -> fp32 residual, RMSNorm of layer 0 into xn (W4 unit order) + group sums
cudaError_t launch_step_begin(const Launch& L, const StepArgs* step, float* r, int D, int32_t* tables,
                              int table_stride, int batch, const __half* gamma, float eps, __half* xn, float* xn_sum);

// ---------------------------------------------------------------- bulk KV store
struct KvStoreArgs {
  const __half* k;  // [L][n][Hkv][d]
  const __half* v;
  int32_t n_tok, n_layers;
  int32_t pos0;        // position of the first appended token
  const int32_t* table;  // this session's block table (device)
  PoolGeom pool;
};
cudaError_t launch_kv_store(const Launch& L, const KvStoreArgs& a);

// ---------------------------------------------------------------- split-K flash-decode attention
struct AttnArgs {
  const __half* qkv;  // [B][qkv_ld]: q (rotated) [Hq d], k (rotated) [Hkv d], v [Hkv d]
  int32_t qkv_ld;
  __half* o;          // [B][ldo] attention output, W4 unit order
  int32_t ldo;
  float* osum;        // [B][ldos] group sums of o (32 dims)
  int32_t ldos;
  int32_t n_heads, n_kv_heads, head_dim;
  int32_t layer;
  int32_t n_split;  // grid.x (<= 64)
  float* part_ml;   // [B][Hkv][n_split][G][2]
  float* part_o;    // [B][Hkv][n_split][G][d]
  uint32_t* counters;  // [B][Hkv]
  PoolGeom pool;
  const StepArgs* step;
};
cudaError_t launch_attention(const Launch& L, const AttnArgs& a, int batch);

// ---------------------------------------------------------------- W4 quantiser (load time)
cudaError_t launch_quantize_w4g32(cudaStream_t s, const float* src, int64_t rows, int64_t cols, uint8_t* codes,
                                  __half2* sm);

}  // namespace mag
