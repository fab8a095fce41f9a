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
enum XSource { XSRC_F16 = 0, XSRC_RESID = 1 };
enum Epilogue { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_STORE_OUT = 3 };
enum TileMap { MAP_PLAIN = 0, MAP_QKV = 1, MAP_SWIGLU = 2 };
constexpr int kTileBytes = 640;  // one 16-row x 64-k tile: 512 B of codes + 128 B of (scale, min)

struct GemvArgs {
  const uint8_t* w;       // tiles [n_mtiles][n_chunks]: W4 640 B, fp16 2048 B each
  int32_t n_mtiles;       // 16-row tiles
  int32_t K;              // reduction length
  int32_t n_chunks;       // ceil(K / 64)
  int32_t chunks_per_cta; // above 4 tokens: k-range of one block, in chunks (W4: a multiple of 4)
  int32_t ks;             // above 4 tokens: k-ranges (fp16 k-split: grid.y; W4: k-windows)
  int32_t tpw;            // fp16 k-split: tiles per warp (1, 2 or 4); a block covers 8 tpw tiles
  int32_t batch;
  // activations: XSRC_F16 fp16 [B][ldx]; XSRC_RESID RMSNorm of the fp32 residual
  const __half* x;
  int32_t ldx;
  float* r;               // fp32 residual [B][ldr] (read by XSRC_RESID, updated by EPI_RESID)
  int32_t ldr;
  float* ss_part;         // per-tile sums of squares [n][16]: written by EPI_RESID, read by XSRC_RESID
  int32_t n_ss;           // XSRC_RESID: entries of ss_part to add up
  const __half* gamma;    // XSRC_RESID gain
  float eps;
  // epilogues
  __half* out_h;          // EPI_QKV [B][ldo] natural, EPI_SWIGLU [B][ldo]
  int32_t ldo;
  int32_t head_dim, n_rot_heads;  // EPI_QKV: heads below n_rot_heads get RoPE
  const float* rope_cos;
  const float* rope_sin;
  float* partial;         // fp16 k-split: [ks][n_mtiles][32][4 * n_tiles]; W4: [n_mtiles][ks][32][4 * n_tiles]
  uint32_t* counters;     // zero between launches (fp16 k-split: per block column; W4: per tile)
  const StepArgs* step;
  // pipelined kernels (up to 4 tokens; W4 above 4 tokens): one block per SM
  int32_t n_cta;          // tile ranges; range i holds tiles [i n_mtiles / n_cta, (i+1) n_mtiles / n_cta)
  int32_t stages;         // ring slots per warp (2..8; W4 above 4 tokens 2..4)
  int32_t t_max;          // most tiles of one range
  uint32_t* err;          // set (bit or) when a pipeline wait gives up
  uint32_t wait_limit;    // polls of a main-loop pipeline wait before it gives up (0: at once)
  // EPI_QKV with an FP16 pool: when kv_store is set, row b's rotated k and its v also go into the pool at
  // (layer, pos[b]) of session sess[b] (heads n_q_heads .. n_q_heads + 2 Hkv of the output)
  int32_t kv_store;
  int32_t n_q_heads;
  int32_t layer;
  PoolGeom pool;
  TraceBuf trace;  // step timeline (debug): block stamps at entry (0), before the wait on the previous
                   // kernel (1), activations staged (2); tag kTraceGemv | n_mtiles << 32 | n_chunks << 8 | B
};

// Polls of a bounded mbarrier wait before it is declared stuck (main-loop default; drain waits always).
constexpr uint32_t kWaitPolls = 1u << 22;
constexpr int kPipeMaxBatch = 4;
size_t gemv_pipe_smem_bytes(int wfmt, int batch, int n_chunks, int stages, int t_max);
int gemv_pipe_max_stages();
size_t gemv_pipe_slot_bytes(int wfmt);  // ring bytes of one slot across the block's warps
cudaError_t launch_gemv_pipe(const Launch& L, const GemvArgs& a, int wfmt, int xsrc, int epi);

// W4 above 4 tokens (k_gemv_batch.cu): grid n_cta tile ranges x ks k-windows of chunks_per_cta chunks.
size_t gemv_batch_smem_bytes(int batch, int cw, int stages, int t_max);
int gemv_batch_max_stages();
size_t gemv_batch_stage_bytes();  // ring bytes of one slot across the block's warps
cudaError_t launch_gemv_batch(const Launch& L, const GemvArgs& a, int xsrc, int epi);

size_t gemv_smem_bytes(const GemvArgs& a, int wfmt);
// Up to 4 tokens: the pipelined kernels; above: W4 k-windows, fp16 (LM head) k-split.
cudaError_t launch_gemv(const Launch& L, const GemvArgs& a, int wfmt, int xsrc, int epi);

// Load-time repack of a W4G32 matrix [N, K] (codes [N][16G] then (scale, min)
// [N][G]) into 640-byte tiles, and back. Tile (mt, c) holds rows
// (r_g, r_g8) for g = 0..7 by `map`: MAP_PLAIN 16 mt + g / +8; MAP_QKV the
// RoPE pair (i, i + d/2) of one head; MAP_SWIGLU gate row 8 mt + g and up row
// F + 8 mt + g.
cudaError_t launch_w4_to_tiles(cudaStream_t s, const uint8_t* canon, int N, int K, int map, int map_arg,
                               uint8_t* tiles);
cudaError_t launch_w4_from_tiles(cudaStream_t s, const uint8_t* tiles, int N, int K, int map, int map_arg,
                                 uint8_t* canon);
// Load-time repack of an fp16 matrix [N, K] (row-major, N % 16 == 0) into
// 2048-byte tiles [N/16][ceil(K/64)]: lane L = (g, t) of a tile holds rows
// g and g+8 at k = 64c + 16t .. 16t+15 (32 bytes each); k >= K is zero.
cudaError_t launch_f16_to_tiles(cudaStream_t s, const __half* src, int N, int K, uint8_t* tiles);
// ---------------------------------------------------------------- chunked prefill (tcgen05)
// Y = X W^T, X fp16 [M][K] by TMA, W read from the decode path's W4 tiles and expanded in shared memory
// (fp16(s q + m)), 128 x 128 tiles. M: tokens, N: GEMM rows (a multiple of 128: the tile rows of 8
// consecutive decode tiles, in the order the epilogue wants). Epilogues: EPI_QKV (fp16 out, q and k
// rotated at position pos0 + row), EPI_RESID (r[row][n] += y), EPI_SWIGLU (out[row][j] = fp16(silu(gate)
// up) from gate and up rows interleaved in blocks of 64).
struct TcGemmArgs {
  int32_t M, N, K;
  int32_t n_valid;  // output columns that exist (RESID: N of the matrix; SWIGLU: F)
  const uint8_t* w;   // the projection's tiles [n_dtiles][C][640]
  int32_t n_dtiles;   // 16-row decode tiles
  int32_t C;          // ceil(K / 64)
  int32_t tpg, gsz, half;  // tile-row map: decode tile j (of 8) row g / g+8 -> GEMM row
                           // (j / tpg) gsz + 8 (j % tpg) + g (+ half)
  float* r;
  int32_t ldr;
  __half* out;
  int32_t ldo;
  int32_t head_dim, n_rot_heads, pos0;
  const int32_t* row_pos;  // when set, row m is rotated at row_pos[m] instead of pos0 + m
  const float* rope_cos;
  const float* rope_sin;
  uint32_t* err;
  uint32_t wait_limit;  // polls of a main-loop wait before it gives up (drains always use kWaitPolls)
  int32_t ksplit;       // 1, or 2: K in halves, merged through part (fp32 partial sums) by the later half
  float* part;          // [blocks][4][2][2][128][32] (tc_gemm_part_floats)
  uint32_t* part_cnt;   // [blocks][4], zero between launches
};
// A 2-D fp16 tensor map over row-major [rows][cols] with 64 x 128 boxes and 128-byte swizzle.
bool make_tmap_2d(void* map_out, const void* base, int64_t rows, int64_t cols);
int tc_gemm_rows_multiple();
// K split of a GEMM of M tokens x N rows x K: 2 when the output blocks fill at most half the SMs
int tc_gemm_ksplit(int M, int N, int K, int n_sm);
size_t tc_gemm_part_floats(int n_sm);  // workspace of a split GEMM
cudaError_t launch_tc_gemm(const Launch& L, const void* map_a, const TcGemmArgs& a, int epi);
cudaError_t launch_rows_to_resid(const Launch& L, const __half* x, float* r, int T, int D);
cudaError_t launch_rmsnorm_rows(const Launch& L, const float* r, const __half* gamma, float eps, int T, int D,
                                __half* xn);
// Rows rows.row[0 .. n) of the fp32 [*][D] src into dst [n][D].
struct RowList {
  int32_t n;
  int32_t row[MAG_MAX_BATCH];
};
cudaError_t launch_gather_rows(const Launch& L, const float* src, int D, const RowList& rows, float* dst);

// ---------------------------------------------------------------- step prologue
// block-table writes, fp16 input -> fp32 residual and its sum of squares (ss_part[0][b])
cudaError_t launch_step_begin(const Launch& L, const StepArgs* step, float* r, int D, int32_t* tables,
                              int table_stride, int batch, float* ss_part);
cudaError_t launch_final_hidden(const Launch& L, const StepArgs* step, const float* r, int D, int batch);

// Debug canaries (MAG_FLAG_DEBUG_CANARY): 64-byte bands of kCanaryByte before and after each arena tensor.
constexpr int kCanaryBand = 64;
constexpr unsigned char kCanaryByte = 0xA5;
struct ArenaCheck {
  const uint8_t* base;
  int32_t n;                    // tensors, at most 16
  uint64_t band[16][2];         // byte offsets of tensor i's band before and after it
  uint32_t* err;                // kErrCanary | 1 << (kErrCanaryShift + i) for a changed band of tensor i
};
cudaError_t launch_arena_check(const Launch& L, const ArenaCheck& a);

// ---------------------------------------------------------------- bulk KV store
struct KvStoreArgs {
  const __half* k;  // [L][n][Hkv][d]
  const __half* v;
  int32_t n_tok, n_layers;
  int32_t pos0;        // position of the first appended token
  const int32_t* table;  // this session's block table (device)
  PoolGeom pool;
  uint32_t* err;         // kErrBounds when a table entry is outside the pool
};
cudaError_t launch_kv_store(const Launch& L, const KvStoreArgs& a);

// Chunked prefill: the rotated k and v of n_tok chunk tokens (rows of the QKV output) stored at
// positions pos0.. of one layer, by the same quantisers.
struct KvChunkArgs {
  const __half* qkv;  // [n_tok][qkv_ld]: q [Hq d], k [Hkv d], v [Hkv d]
  int32_t qkv_ld, n_heads;
  int32_t n_tok, pos0, layer;
  const int32_t* table;
  PoolGeom pool;
  // when set, pos0 and the table row are read on the device from the step arguments (session sess[0] from
  // position pos[0]), so a captured graph serves any session and position
  const StepArgs* step;
  // when set (several sessions in one chunk), token t goes to session row_sess[t] at position row_pos[t]
  const int32_t* row_pos;
  const int32_t* row_sess;
  uint32_t* err;  // kErrBounds when a table entry is outside the pool
};
cudaError_t launch_kv_store_chunk(const Launch& L, const KvChunkArgs& a);

// Chunked prefill: causal GQA attention of the chunk's queries (token t at position pos0 + t) over the
// pool positions 0 .. pos0 + t (the chunk's own keys stored first). Pool values are widened to fp16 in
// shared memory (exact for FP16 storage).
// One session's tokens in a chunk: rows row0 .. row0 + n_tok - 1 of the QKV output, at positions pos0 ..
struct PfSeg {
  int32_t row0, n_tok, pos0, sess;
};
struct PrefillAttnArgs {
  const __half* qkv;  // [rows][qkv_ld]
  int32_t qkv_ld;
  __half* o;          // [rows][ldo]
  int32_t ldo;
  int32_t n_heads, n_kv_heads, head_dim, layer;
  PoolGeom pool;      // block tables of the sessions in pool.tables
  int32_t n_seg;      // grid.z
  PfSeg seg[MAG_MAX_BATCH];
  uint32_t* err;      // kErrBounds when a table entry is outside the pool
};
cudaError_t launch_prefill_attention(const Launch& L, const PrefillAttnArgs& a);

// ---------------------------------------------------------------- split-K flash-decode attention
struct AttnArgs {
  const __half* qkv;  // [B][qkv_ld]: q (rotated) [Hq d], k (rotated) [Hkv d], v [Hkv d]
  int32_t qkv_ld;
  __half* o;          // [B][ldo] attention output
  int32_t ldo;
  int32_t n_heads, n_kv_heads, head_dim;
  int32_t layer;
  int32_t n_split;   // cluster size (<= 16)
  int32_t n_groups;  // clusters per (session, KV head), 1..kAttnMaxGroups: grid.x = n_split * n_groups
  // n_groups > 1: per (session, KV head, cluster) the cluster's (m, l, o) of the G d outputs, fp32
  // [B][Hkv][kAttnMaxGroups][3][G d], and per (session, KV head) a counter of arrived blocks (zero between
  // launches: the last block to arrive merges and resets it)
  float* part;
  uint32_t* arrivals;
  PoolGeom pool;
  const StepArgs* step;
  // 0: row b appends its own token (position pos[b]) and attends to 0 .. pos[b].
  // 1: the rows are consecutive new tokens of one session (pos[b] = pos[0] + b) whose keys and values an
  //    earlier kernel stored; row b attends causally to 0 .. pos[b] and appends nothing.
  // 2: as 0, but the QKV projection already stored row b's own key and value in the pool.
  int32_t stored;
  // 0: 4 warps per block (two blocks per SM); 1: the wide variant, 8 warps per block at head_dim 128
  // (16 at 64), one block per SM, for long contexts
  int32_t wide;
  uint32_t* err;  // kErrBounds when a table entry is outside the pool
  TraceBuf trace;  // step timeline (debug): stamps at entry (0), after the wait (1), keys done (2), end (3);
                   // tag kTraceAttn | layer
};
cudaError_t launch_attention(const Launch& L, const AttnArgs& a, int batch);
constexpr int kAttnMaxGroups = 8;
// Largest split count (cluster size) the device can co-schedule for this head size, KV type and variant.
cudaError_t attention_max_cluster(int head_dim, int kv_dtype, bool wide, int* out);

// ---------------------------------------------------------------- W4 quantiser (load time)
cudaError_t launch_quantize_w4g32(cudaStream_t s, const float* src, int64_t rows, int64_t cols, uint8_t* codes,
                                  __half2* sm);

}  // namespace mag
