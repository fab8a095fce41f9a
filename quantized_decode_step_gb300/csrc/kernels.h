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
enum XMode { X_F16 = 0, X_NORM = 1 };
enum Epilogue { EPI_STORE = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_STORE_OUT = 3 };

struct GemvArgs {
  const uint8_t* w;       // W4 codes [N][w_row_bytes] or fp16 [N][K]
  const __half2* sm;      // W4 (scale, min) pairs [N][sm_row]
  int64_t w_row_bytes;
  int32_t sm_row;         // groups per row (W4)
  int32_t n_mtiles;       // m-tiles of 16 output rows (SwiGLU: 8 gate + 8 up rows)
  int32_t swiglu_f;       // SwiGLU: F (up rows start at F)
  int32_t K;              // reduction length
  int32_t n_chunks;       // ceil(K / 64)
  int32_t chunks_per_cta; // k-range of one block, in 64-wide chunks
  int32_t ks;             // k-splits (grid.y)
  int32_t mpc;            // m-tiles per block
  int32_t wk;             // warps sharing one m-tile's k-range
  const __half* x;        // X_F16: [B][ldx]
  int32_t ldx;
  const float* r;         // X_NORM: residual [B][ldr] and gain [K]
  int32_t ldr;
  const __half* gamma;
  float eps;
  int32_t batch;
  __half* out_h;          // EPI_STORE / EPI_SWIGLU: [B][ldo]
  float* out_r;           // EPI_RESID: [B][ldo] (+=)
  int32_t ldo;
  float* partial;         // ks > 1: [ks][n_mtiles][32][4 * n_tiles]
  uint32_t* counters;     // ks > 1: [grid.x], zero between launches
  const StepArgs* step;   // EPI_STORE_OUT: output pointer of the step
};

size_t gemv_smem_bytes(const GemvArgs& a, int n_tok_tiles);
cudaError_t launch_gemv(const Launch& L, const GemvArgs& a, int wfmt, int xmode, int epi);

// ---------------------------------------------------------------- step prologue
cudaError_t launch_step_begin(const Launch& L, const StepArgs* step, float* r, int D, int32_t* tables,
                              int table_stride, int batch);
cudaError_t launch_final_hidden(const Launch& L, const StepArgs* step, const float* r, int D, int batch);

// ---------------------------------------------------------------- RoPE + KV append, bulk KV store
struct RopeAppendArgs {
  const __half* qkv;  // [B][(Hq+2Hkv)d]
  __half* q_out;      // [B][Hq d] rotated
  const float* rope_cos;  // [max_pos][d/2]
  const float* rope_sin;
  int32_t n_heads, n_kv_heads, head_dim;
  int32_t layer;
  PoolGeom pool;
  const StepArgs* step;
};
cudaError_t launch_rope_append(const Launch& L, const RopeAppendArgs& a, int batch);

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
  const __half* q;  // [B][Hq d] rotated
  __half* o;        // [B][Hq d]
  int32_t n_heads, n_kv_heads, head_dim;
  int32_t layer;
  int32_t n_split;  // grid.x
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
