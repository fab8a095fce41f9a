/*
 * Oracle for the quantized decode step -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU implementation of what the decode
 * step computes. Only the tests, the smoke check and the bench's CPU-baseline
 * leg may load it; the product library never calls it and shares no code,
 * header, table or helper with it.
 *
 * Sources (pages, cited by title and section):
 *   [Magnitude]   "Magnitude: on-device AI-agent inference engine --
 *                 self-optimising scheduling and elastic memory pools"
 *                 (0539edu.com), sections 3.2, 4.3, 5.1, 5.2
 *   [Core]        "5. Core modules: format, runtime, scheduling, memory and
 *                 routing" (ai-infra.cypggs.com), sections 5.1, 5.2, 5.4
 *   [TFLite]      "TFLite memory planner" (pwwt.cn), sections 2.1-2.3, 3.2
 *
 * Precision: the pages fix 4-bit weights with FP16 activations ([Core] 5.1,
 * "W4A16"), so every value the step hands from one operation to the next is
 * rounded to fp16 at the same cast points the GPU has; everything in between
 * is carried in double. Quantisation decisions (4-bit and INT8 codes) are
 * taken in fp32 with IEEE division and round-half-even, as the format defines.
 *
 * Parity pins: every function here is pinned by a test in tests/ against
 * closed forms, invariants, worked examples or library routines. The step is
 * orc_layer per layer then orc_output; its composition is pinned against
 * models built from torch library routines: one layer, two chained layers
 * with their own weights and caches, and the LM-head output; several
 * sequences in one pass are pinned to the same sequences run one by one.
 */
#ifndef MAG_ORACLE_H
#define MAG_ORACLE_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_KV_FP16 = 0, ORC_KV_INT8 = 1, ORC_KV_INT4 = 2 };

typedef struct {
  int n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab; /* vocab 0: output the hidden state */
  float rms_eps;
  float rope_base;
  int kv_dtype;
  int block_tokens;
} orc_cfg;

/* W4 g32 packed tensors in the canonical format (see orc_w4g32_quantize). */
typedef struct {
  const uint8_t* const* wqkv;  /* [L] -> u8 [(Hq+2Hkv)d][D/2] */
  const uint16_t* const* sqkv; /* [L] -> fp16 pairs [(Hq+2Hkv)d][D/32][2] = (scale, min) */
  const uint8_t* const* wo;
  const uint16_t* const* so;
  const uint8_t* const* wgu; /* rows [gate F; up F] */
  const uint16_t* const* sgu;
  const uint8_t* const* wdown;
  const uint16_t* const* sdown;
  const uint16_t* const* gamma1; /* [L] -> fp16 [D] */
  const uint16_t* const* gamma2;
  const uint16_t* gamma_f; /* fp16 [D] */
  const uint16_t* lm_head; /* fp16 [V][D] or NULL when vocab == 0 */
} orc_weights;

typedef struct orc_kv orc_kv;

/* ---- threads of the parallel loops (n < 1: every core); returns the count in use ---- */
int orc_set_threads(int n);

/* ---- fp16 ---- */
uint16_t orc_f64_to_f16(double x);
uint16_t orc_f32_to_f16(float x);
float orc_f16_to_f32(uint16_t h);
void orc_f32_to_f16_array(const float* x, int64_t n, uint16_t* out);

/* ---- 4-bit group-32 weights ---- */
void orc_w4g32_quantize(const float* w, int64_t n_rows, int64_t n_cols, uint8_t* packed, uint16_t* sm);
void orc_w4g32_dequant(const uint8_t* packed, const uint16_t* sm, int64_t n_rows, int64_t n_cols, float* out);
void orc_w4_gemv(const uint8_t* packed, const uint16_t* sm, int64_t n_rows, int64_t n_cols, int n_tok,
                 const uint16_t* x_f16, double* y);
void orc_w4_gemv_folded(const uint8_t* packed, const uint16_t* sm, int64_t n_rows, int64_t n_cols,
                        const uint16_t* x_f16, double* y);

/* ---- KV quantisers ---- */
void orc_kv_quant_int8(const uint16_t* x_f16, int n_vec, int d, int8_t* q, uint16_t* scale);
void orc_kv_quant_int4(const uint16_t* x_f16, int n_vec, int d, uint8_t* packed, uint16_t* sm);

/* ---- block pool layout and allocator model ---- */
int64_t orc_kv_block_bytes(int n_kv_heads, int head_dim, int kv_dtype, int block_tokens);
int64_t orc_kv_offset(int n_kv_heads, int head_dim, int kv_dtype, int block_tokens, int64_t pool_blocks,
                      int layer, int64_t block, int part, int head, int slot);
int64_t orc_kv_bytes_per_token(int n_layers, int n_kv_heads, int head_dim, double bytes_per_value);
int64_t orc_kv_max_context(double total_bytes, double os_bytes, double weight_bytes, double kv_bytes_per_token);

/* ---- arena planner ---- */
int64_t orc_arena_plan(int n, const int64_t* size, const int* first, const int* last, int64_t align,
                       int closed_intervals, int64_t* offset);

/* ---- layer pieces ---- */
void orc_rmsnorm(const double* r, const uint16_t* gamma, int n, float eps, uint16_t* out);
void orc_rope_table(int max_pos, int head_dim, float base, float* cos_out, float* sin_out);
void orc_rope_apply(const uint16_t* x, int head_dim, const float* cos_row, const float* sin_row, uint16_t* out);

/* ---- logical KV store (per session) ---- */
orc_kv* orc_kv_create(const orc_cfg* cfg, int capacity);
void orc_kv_destroy(orc_kv* kv);
int orc_kv_len(const orc_kv* kv);
void orc_kv_truncate(orc_kv* kv, int len);
int orc_kv_commit(orc_kv* kv, int n);
int orc_kv_append(orc_kv* kv, int n_tok, const uint16_t* k_f16, const uint16_t* v_f16); /* [L][n][Hkv][d] */
void orc_kv_read(const orc_kv* kv, int layer, int which, int tok, int head, float* out);
int64_t orc_kv_stored(const orc_kv* kv, int layer, int which, int tok, int head, uint8_t* data, uint8_t* meta);
void orc_attention(const orc_cfg* cfg, const orc_kv* kv, int layer, int kv_head, const uint16_t* q_f16, int n_keys,
                   uint16_t* out_f16);

/* ---- whole step ---- */
int orc_layer(const orc_cfg* cfg, const orc_weights* w, int layer, int n_seq, orc_kv* const* kv, const int* n_tok,
              const double* r_in, const float* rope_cos, const float* rope_sin, int rope_rows, double* r_out);
void orc_output(const orc_cfg* cfg, const orc_weights* w, const double* r, uint16_t* out_f16);
int orc_forward(const orc_cfg* cfg, const orc_weights* w, int n_seq, orc_kv* const* kv, const int* n_tok,
                const uint16_t* x_f16, const float* rope_cos, const float* rope_sin, int rope_rows,
                uint16_t* out_f16);

#ifdef __cplusplus
}
#endif
#endif
